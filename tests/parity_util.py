"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
(binding) and the oracle on the same seeded inputs, compare."""
import numpy as np
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads

# GEMM tolerance: the method's statement of the target is "max relative error
# <= 1e-3 against the FP64 accumulation of identical dequantised operands",
# read normwise (max |C - R| / max |R|) because an elementwise ratio is
# unbounded where R cancels to ~0.  BF16 output adds one BF16 rounding (half
# an ulp) on top.
GEMM_TOL = 1e-3

# Elementwise bound of the FP32 result, on top of the normwise one:
#   |C - R| <= 1e-3 |R| + K 2^-24 S,   S = (T_A T_B) sum_k |(e s)_a| |(e s)_b|,
# K 2^-24 S being the classical bound of binary32 summation of the K exact
# products in any order.  It scales with each element's own operands, so a
# large error on a row of tiny magnitude (a dgrad row of a 1e-8 gradient)
# cannot hide below the largest entries of the matrix.  Over the entries
# where the second term is below the first (|R| > 1e3 K 2^-24 S: no heavy
# cancellation) it is a relative error of at most 2e-3; the largest relative
# error there is reported.
def gemm_abs_reference(pa, sa, pb, sb, alpha, fmt=0):
    """S = alpha |deq(A)| |deq(B)|^T from the oracle's exact e*s operands."""
    return alpha * (np.abs(oracle.deq_es(pa, sa, fmt)) @ np.abs(oracle.deq_es(pb, sb, fmt)).T)


def check_gemm_elementwise(C, R, S, K) -> float:
    C = np.asarray(C, np.float64)
    err = np.abs(C - R)
    floor = K * 2.0 ** -24 * S
    bad = err > GEMM_TOL * np.abs(R) + floor
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{int(bad.sum())} elements beyond 1e-3|R| + K 2^-24 S; first {i}: "
                             f"C={C[i]!r} R={R[i]!r} S={S[i]!r}")
    well = np.abs(R) > floor / GEMM_TOL
    return float((err[well] / np.abs(R[well])).max()) if well.any() else 0.0


def check_gemm_bf16(C16, R):
    """The BF16 result within one BF16 ulp of R plus 1e-3 max |R|, elementwise."""
    C16 = np.asarray(C16, np.float64)
    bound = bf16_ulp(R) + GEMM_TOL * np.abs(R).max()
    bad = np.abs(C16 - R) > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{int(bad.sum())} BF16 elements beyond ulp + 1e-3 max|R|; first {i}: "
                             f"C={C16[i]!r} R={R[i]!r}")


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return workloads.to_torch_bf16(bits).cuda()


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def gpu_tensor_scale(x: torch.Tensor, fmt=0, headroom=1.0):
    from fp4_block_scaled_bf16_gb300 import fp4q
    a = fp4q.amax(x)
    return a, fp4q.tensor_scale(a, fmt, headroom)


def check_quantize(bits: np.ndarray, axis: int, fmt=0, rnd=0, seed=0, T=None, headroom=1.0):
    """Quantise on the GPU and with the oracle; assert bytes, stats and the
    fused amax agree exactly.  Returns the oracle outputs."""
    from fp4_block_scaled_bf16_gb300 import fp4q
    x = to_dev(bits)
    if T is None:
        a_dev, T_dev = gpu_tensor_scale(x, fmt, headroom)
        a_or, _ = oracle.amax(bits)
        T_or = oracle.tensor_scale(a_or, fmt, headroom)
        assert float(a_dev.item()) == a_or
        assert float(T_dev.item()) == T_or
    else:
        T_dev = torch.tensor([T], dtype=torch.float32, device="cuda")
        T_or = float(np.float32(T))
    q = fp4q.quantize(x, axis, T_dev, fmt, rnd, seed, stats=True, want_amax=True)
    torch.cuda.synchronize()
    out = {}
    axes = [oracle.ROW, oracle.COL] if axis == fp4q.AXIS_BOTH else [axis]
    for k, ax in enumerate(axes):
        p, s, st = oracle.quantize(bits, ax, T_or, fmt, rnd, seed)
        gp = q.payload_row if ax == oracle.ROW else q.payload_col
        gs = q.scales_row if ax == oracle.ROW else q.scales_col
        gp, gs = np_u8(gp), np_u8(gs)
        if not np.array_equal(gp, p):
            bad = np.argwhere(gp != p)
            raise AssertionError(f"payload axis {ax}: {len(bad)} bytes differ, first {bad[:4].tolist()} "
                                 f"gpu {gp[tuple(bad[0])]:#04x} oracle {p[tuple(bad[0])]:#04x}")
        if not np.array_equal(gs, s):
            bad = np.argwhere(gs != s)
            raise AssertionError(f"scales axis {ax}: {len(bad)} differ, first {bad[:4].tolist()}")
        gst = q.stats.cpu().numpy()[k].astype(np.uint64)
        assert np.array_equal(gst, st), (ax, gst, st)
        out[ax] = (p, s, st)
    assert float(q.amax.item()) == oracle.amax(bits)[0]
    return out, T_or, q


def gemm_error(C: np.ndarray, R: np.ndarray) -> float:
    return float(np.abs(C.astype(np.float64) - R).max() / max(np.abs(R).max(), 1e-300))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def sampled_check(A, B, Cdev32, rows, cols, fmt=0):
    """Full row and column stripes of the reference via the oracle's exact
    e*s operands and a binary64 matmul: the normwise error over the stripes
    (returned) and the elementwise bound on every entry of them."""
    pa, sa = A[0].cpu().numpy(), A[1].cpu().numpy()
    pb, sb = B[0].cpu().numpy(), B[1].cpu().numpy()
    alpha = float(A[2].item()) * float(B[2].item())
    K = pa.shape[1] * 2
    C = Cdev32
    ea_r, eb = oracle.deq_es(pa[rows], sa[rows], fmt), oracle.deq_es(pb, sb, fmt)
    R_rows, S_rows = alpha * (ea_r @ eb.T), alpha * (np.abs(ea_r) @ np.abs(eb).T)
    del ea_r, eb
    ea, eb_c = oracle.deq_es(pa, sa, fmt), oracle.deq_es(pb[cols], sb[cols], fmt)
    R_cols, S_cols = alpha * (ea @ eb_c.T), alpha * (np.abs(ea) @ np.abs(eb_c).T)
    del ea, eb_c
    c_rows = C[torch.from_numpy(rows).to(C.device)].cpu().numpy().astype(np.float64)
    c_cols = C[:, torch.from_numpy(cols).to(C.device)].cpu().numpy().astype(np.float64)
    check_gemm_elementwise(c_rows, R_rows, S_rows, K)
    check_gemm_elementwise(c_cols, R_cols, S_cols, K)
    scale = max(np.abs(R_rows).max(), np.abs(R_cols).max())
    e1 = np.abs(c_rows - R_rows).max() / scale
    e2 = np.abs(c_cols - R_cols).max() / scale
    return max(e1, e2)


def stripes(n, rng, tile):
    s = list(range(0, min(tile, n))) + list(range(max(n - tile, 0), n))
    s += list(rng.choice(n, 64, replace=False))
    return np.unique(np.array(s))


def extreme_rows(bits: np.ndarray, k: int = 4) -> np.ndarray:
    """The k rows of a BF16 matrix with the largest and the k with the
    smallest non-zero row amax (a dgrad's rows of extreme gradient
    magnitude, where a scale or factor error would hide below the rest)."""
    a = np.abs(workloads.bf16_bits_to_f32(bits)).max(axis=1)
    order = np.argsort(a)
    nz = order[a[order] > 0]
    return np.unique(np.r_[nz[:k], nz[-k:]])

