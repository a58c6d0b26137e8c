"""The int8 KV cache of a prompt-attention workload, written twice from the
same fp32 rows: on the host by the oracle's per-token quantiser and on the
device by the library's int8kv_cache_write.  The attention parity tests give
each side its own cache and check first that the two are the same bytes."""

import numpy as np

import oracle


def oracle_cache(x: dict) -> dict:
    """q bits plus int8 codes [Hkv, Nk, 128] and fp16 scales [Hkv, Nk] from the oracle."""
    out = {"q": x["q"]}
    for key in ("k", "v"):
        codes, bits = oracle.cache_quantise(x[key + "_raw"])
        out[key] = codes
        out[key + "_scale"] = bits.view(np.float16)
    return out


def device_cache(qas, x: dict):
    """(q, k codes, k scales, v codes, v scales) on the GPU, the cache written by
    int8kv_cache_write from the token-major view of the rows."""
    import torch

    q = torch.from_numpy(np.ascontiguousarray(x["q"]).view(np.int16)).view(torch.bfloat16).cuda()
    k = torch.from_numpy(x["k_raw"]).cuda().permute(1, 0, 2)  # [Nk, Hkv, 128] view
    v = torch.from_numpy(x["v_raw"]).cuda().permute(1, 0, 2)
    hkv, nk, d = x["k_raw"].shape
    kc = torch.empty((hkv, nk, d), dtype=torch.int8, device="cuda")
    vc = torch.empty_like(kc)
    ks = torch.empty((hkv, nk), dtype=torch.float16, device="cuda")
    vs = torch.empty_like(ks)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qas.int8kv_cache_write(k, v, kc, ks, vc, vs, 0, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return q, kc, ks, vc, vs


def both_caches(qas, x: dict):
    """The oracle's cache (host dict) and the device tensors, checked bit for bit."""
    host = oracle_cache(x)
    q, kc, ks, vc, vs = device_cache(qas, x)
    assert np.array_equal(kc.cpu().numpy(), host["k"]) and np.array_equal(vc.cpu().numpy(), host["v"])
    assert np.array_equal(ks.cpu().numpy().view(np.uint16), host["k_scale"].view(np.uint16))
    assert np.array_equal(vs.cpu().numpy().view(np.uint16), host["v_scale"].view(np.uint16))
    return host, (q, kc, ks, vc, vs)
