"""Helpers shared by the GPU parity tests (device inputs, tolerances)."""
import numpy as np
import torch

DEV = torch.device("cuda:0")

# Agreement rules.  fp32 path: max-abs 1e-5.  bf16 path: max-abs 2e-2 and
# mean-rel 2e-3 (sum|a-b| / sum|b|) against the fp64 oracle on the same
# bf16-rounded inputs.  Indexer scores of the bf16 path are fp32 results of
# exact bf16 products summed in fp32: 128 products of two unit normals per
# index head (sum of magnitudes ~80, rounding ~80 * 2^-24 per add in the worst
# order), then 64 ReLUs weighted by w ~ N(0, 1/64).  The measured error is a
# few 1e-5; the bound below is about ten times that and half the 1e-3 band
# inside which end-to-end index sets may differ (near ties), so a score error
# can never by itself move a key across that band.
FP32_TOL = 1e-5
BF16_MAXABS, BF16_MEANREL = 2e-2, 2e-3
SCORE_MAXABS = 5e-4
NEAR_TIE = 1e-3


def lib():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_long_gb300 as dsa
    return dsa


def params(dsa, wl, **kw):
    base = dict(B=wl["B"], S_q=wl["S"], S_k=wl["S"], H=wl["H"], d_qk=wl["d_qk"], d_v=wl["d_v"],
                H_I=wl["H_I"], d_I=wl["d_I"], topk=wl["topk"], scale=wl["scale"], dtype=wl["dtype"])
    base.update(kw)
    return dsa.make_params(**base)


def np64(t):
    return t.detach().to("cpu").double().numpy()


def bf16_close(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    d = np.abs(got - ref)
    maxabs = float(d.max()) if d.size else 0.0
    meanrel = float(d.sum() / max(np.abs(ref).sum(), 1e-300))
    return maxabs <= BF16_MAXABS and meanrel <= BF16_MEANREL, maxabs, meanrel


def near_tie_violations(idx_gpu, idx_ref, scores_ref, k, tol=NEAR_TIE):
    """Keys in the symmetric difference of two index rows whose oracle score is
    farther than tol from the row's k-th largest oracle score."""
    bad = []
    for r in range(idx_gpu.shape[0]):
        a = set(int(x) for x in idx_gpu[r] if x >= 0)
        b = set(int(x) for x in idx_ref[r] if x >= 0)
        if a == b:
            continue
        row = scores_ref[r]
        fin = np.sort(row[np.isfinite(row)])[::-1]
        kth = fin[min(k, fin.size) - 1]
        for s in a ^ b:
            if abs(row[s] - kth) > tol:
                bad.append((r, s, float(row[s]), float(kth)))
    return bad


def empty_outputs(wl, S_q, dtype):
    B, H, d_v, k = wl["B"], wl["H"], wl["d_v"], wl["topk"]
    return dict(idx=torch.empty(B, S_q, k, dtype=torch.int32, device=DEV),
                out=torch.empty(B, S_q, H, d_v, dtype=dtype, device=DEV),
                m=torch.empty(B, S_q, H, device=DEV), l=torch.empty(B, S_q, H, device=DEV))
