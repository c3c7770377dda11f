"""Shared helpers for the GPU parity tests: tolerances and comparisons against
the fp64 oracle. The oracle never sees anything the CUDA library produced
except the page set it is asked to verify (the sparse attention output is
evaluated over the selection the GPU made, once that selection has been checked
against the oracle's own top-K)."""
import numpy as np
import torch

# Attention output tolerance vs fp64: fp16 I/O, fp32 accumulation.
MAX_ABS = 2e-3
MEAN_ABS = 2e-4
# Top-K: pages whose oracle score is within this relative distance of the
# K-th score may fall on either side of the cut.
TOPK_REL = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_attn_close(got: torch.Tensor, ref: np.ndarray, what: str = "out"):
    g = to64(got)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3e} > {MAX_ABS}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e} > {MEAN_ABS}"
    return err.max(), err.mean()


def check_topk(gpu_idx: np.ndarray, ref_scores: np.ndarray, valid_len, S: int, K: int):
    """Selected sets equal the oracle's up to near-ties at the K-th score."""
    B, Hkv, _ = gpu_idx.shape
    exempted = 0
    for b in range(B):
        P = (int(valid_len[b]) + S - 1) // S
        n = min(K, P)
        for h in range(Hkv):
            row = gpu_idx[b, h]
            assert np.all(row[n:] == -1), f"padding wrong at b={b} h={h}"
            sel = row[:n]
            assert np.all(sel >= 0) and np.all(sel < P), f"index out of range at b={b} h={h}"
            assert np.all(np.diff(sel) > 0), f"not ascending/distinct at b={b} h={h}"
            if P <= K:
                assert np.array_equal(sel, np.arange(P))
                continue
            sc = ref_scores[b, h, :P]
            order = np.lexsort((np.arange(P), -sc))
            kth = sc[order[K - 1]]
            exempt = np.abs(sc - kth) <= TOPK_REL * abs(kth)
            ref_set = np.zeros(P, bool); ref_set[order[:K]] = True
            got_set = np.zeros(P, bool); got_set[sel] = True
            bad = (ref_set != got_set) & ~exempt
            assert not bad.any(), f"b={b} h={h}: pages {np.nonzero(bad)[0][:10]} differ outside the tie window"
            exempted += int(((ref_set != got_set) & exempt).sum())
    return exempted


def score_tolerance(q64: np.ndarray, meta64: np.ndarray, G: int) -> np.ndarray:
    """Bound on |fp32 - fp64| for U: at most ~20 rounded additions deep, so
    2^-17 times the sum of |terms| is a safe ceiling."""
    B, Hq, D = q64.shape
    Hkv = Hq // G
    qa = np.abs(q64).reshape(B, Hkv, G, D)
    mag = np.maximum(np.abs(meta64[:, :, :, 0, :]), np.abs(meta64[:, :, :, 1, :]))  # [B,Hkv,P,D]
    tot = np.einsum("bkgd,bkpd->bkgp", qa, np.nan_to_num(mag)).max(axis=2)
    return tot * 2.0 ** -17 + 1e-30
