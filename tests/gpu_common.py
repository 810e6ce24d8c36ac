"""Helpers shared by the GPU tests: oracle comparison with the attention tolerance."""
import numpy as np
import torch

from oracle import attend as OA

# Attention tolerance: max-abs 2e-3 and relative-L2 1e-2 on the output (bf16 in,
# fp32 accumulate).  lse: fp32 running sums over <= 2^20 keys with bf16-rounded
# weights; |error| <= 2e-3 holds with a wide margin (the observed error is ~1e-5).
MAX_ABS = 2e-3
REL_L2 = 1e-2
LSE_ABS = 2e-3


def compare(w, out, lse, items_per_stream=None, cache=0, threads=None, fp8=False):
    """Compare device outputs [S][R][H][512] / [S][R][H] against the fp64 oracle."""
    ref = OA.attend_workload(w, cache=cache, items_per_stream=items_per_stream, threads=threads, fp8=fp8)
    o = out.float().cpu().numpy().reshape(w.S, w.R * w.H, 512)
    lz = lse.float().cpu().numpy().reshape(w.S, w.R * w.H)
    worst = dict(max_abs=0.0, rel_l2=0.0, lse=0.0)
    for s, (items, o_ref, l_ref) in enumerate(ref):
        if len(items) == 0:
            continue
        got = o[s, items].astype(np.float64)
        assert np.all(np.isfinite(got)), f"stream {s}: non-finite output"
        ma = float(np.max(np.abs(got - o_ref)))
        rl = float(np.linalg.norm(got - o_ref) / max(np.linalg.norm(o_ref), 1e-30))
        le = float(np.max(np.abs(lz[s, items] - l_ref)))
        worst["max_abs"] = max(worst["max_abs"], ma)
        worst["rel_l2"] = max(worst["rel_l2"], rl)
        worst["lse"] = max(worst["lse"], le)
        assert ma <= MAX_ABS, f"stream {s}: max-abs {ma:.3e} > {MAX_ABS}"
        assert rl <= REL_L2, f"stream {s}: rel-L2 {rl:.3e} > {REL_L2}"
        assert le <= LSE_ABS, f"stream {s}: lse error {le:.3e} > {LSE_ABS}"
    return worst


def no_device_error(pool):
    rc, detail = pool.last_error()
    assert rc == 0, f"device error word: {rc} (detail {detail})"


def sample_items(w, per_stream: int, seed: int = 0, long_threshold: int = 1 << 30):
    """A seeded sample of r*H+h items for every stream (all items when few)."""
    g = np.random.default_rng(seed)
    res = []
    for s in range(w.S):
        n = w.R * w.H
        k = per_stream if int(w.lens[s]) * n > long_threshold or n > per_stream else n
        k = min(k, n)
        items = np.sort(g.choice(n, size=k, replace=False)).astype(np.int32)
        # always include both ends
        items = np.unique(np.concatenate([items, [0, n - 1]])).astype(np.int32)
        res.append(items)
    return res


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
