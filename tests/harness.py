"""Shared helpers of the GPU tests: run the engine through its binding, run
the oracle on the same inputs, compare with the stated tolerances.

Tolerances against the fp64 oracle:
  * outputs: relative Frobenius error <= 2e-3 per (sequence, value head),
    over that head's [tokens, dv] block, wherever the block holds at least
    1,024 elements.  A shorter block (a one-token decode: 128 elements) is
    too small for the bound: bf16 rounding alone costs ~1.7e-3 relative (rms)
    with a spread that grows as the block shrinks, so there the norm runs over
    the sequence's whole [tokens, heads, dv] output instead.  In addition the
    error beyond the output format must stay <= 1e-3 over the same blocks: per
    element, the part of |o - oracle| that exceeds half a unit in the last
    place of the output dtype at the oracle's value (a correctly rounded
    fp64 value is within half an ulp of it, so only the kernel's own error
    shows), as a relative Frobenius norm.
  * states: relative Frobenius error <= 1e-4 per (sequence, value head) over
    the dv x dk matrix (fp32 storage, no format loss).
  * conv windows, page indexing and checkpoint placement: exact.

Every check records its worst value; the session prints the worst margin of
each test at its end (tests/conftest.py).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import gated_deltanet_state_gb300 as gdn
from gated_deltanet_state_gb300 import inputs

OUT_TOL = 2e-3
OUT_FORMAT_TOL = 1e-3
STATE_TOL = 1e-4
HEAD_BLOCK_MIN = 1024     # elements of a (sequence, head) block checked on its own

# (test id, quantity, worst value, tolerance) of every check in this process
MARGINS: list[tuple[str, str, float, float]] = []


def _record(kind: str, worst: float, tol: float) -> None:
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    MARGINS.append((test, kind, float(worst), float(tol)))


def dims(shape) -> oracle.Dims:
    return oracle.Dims(shape.num_qk_heads, shape.num_v_heads, shape.head_dim_k, shape.head_dim_v,
                       shape.q_scale, shape.norm_eps)


def rel_fro(x, ref, axis) -> np.ndarray:
    """Relative Frobenius error reduced over `axis` (the rest is kept)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.sqrt(((x - ref) ** 2).sum(axis=axis))
    den = np.sqrt((ref ** 2).sum(axis=axis))
    return num / np.maximum(den, 1e-30)


def round_to(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """The oracle's values rounded to the engine's output dtype."""
    return torch.from_numpy(np.ascontiguousarray(ref)).to(dtype).double().numpy()


def ulp_of(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """One unit in the last place of `dtype` at each value of ref."""
    mant = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}.get(dtype, 52)
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - mant), 0.0)


def out_errors(o_gpu, o_ref, cu, head_block_min=HEAD_BLOCK_MIN):
    """Worst (plain, format-aware) relative Frobenius errors of outputs laid
    out [rows, ..., heads, dv], sequences delimited along the rows by cu.

    A sequence's outputs are compared head by head when a head's block
    ([rows, ..., dv] of that head) holds at least `head_block_min` elements,
    else as one block over all its heads."""
    dt = o_gpu.dtype if hasattr(o_gpu, "dtype") and isinstance(o_gpu.dtype, torch.dtype) else torch.float32
    o = o_gpu.double().cpu().numpy() if hasattr(o_gpu, "cpu") else np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64).reshape(o.shape)
    beyond = np.maximum(np.abs(o - o_ref) - 0.5 * ulp_of(o_ref, dt), 0.0)
    H, D = o.shape[-2], o.shape[-1]
    plain = fmt = 0.0
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b == a:
            continue
        ref = o_ref[a:b].reshape(-1, H, D)
        diff = (o[a:b] - o_ref[a:b]).reshape(-1, H, D)
        bey = beyond[a:b].reshape(-1, H, D)
        if ref.shape[0] * D >= head_block_min:
            den = np.maximum(np.sqrt((ref ** 2).sum(axis=(0, 2))), 1e-30)
            plain = max(plain, float(np.max(np.sqrt((diff ** 2).sum(axis=(0, 2))) / den)))
            fmt = max(fmt, float(np.max(np.sqrt((bey ** 2).sum(axis=(0, 2))) / den)))
        else:
            den = max(float(np.linalg.norm(ref)), 1e-30)
            plain = max(plain, float(np.linalg.norm(diff)) / den)
            fmt = max(fmt, float(np.linalg.norm(bey)) / den)
    return plain, fmt


def assert_out_close(o_gpu, o_ref, cu, tol=OUT_TOL, fmt_tol=OUT_FORMAT_TOL):
    plain, fmt = out_errors(o_gpu, o_ref, cu)
    _record("out", plain, tol)
    _record("out_beyond_half_ulp", fmt, fmt_tol)
    assert plain <= tol, f"output rel. Frobenius error {plain:.3e} > {tol:.1e}"
    assert fmt <= fmt_tol, f"output error beyond half an ulp of the output format {fmt:.3e} > {fmt_tol:.1e}"
    return plain


def assert_state_close(S_gpu, S_ref, tol=STATE_TOL):
    """S [..., Hv, dv, dk]: per head over (dv, dk)."""
    S_gpu = S_gpu.float().cpu().numpy() if hasattr(S_gpu, "cpu") else S_gpu
    e = rel_fro(S_gpu, S_ref, axis=(-2, -1))
    worst = float(np.max(e)) if e.size else 0.0
    _record("state", worst, tol)
    assert worst <= tol, f"state rel. Frobenius error {worst:.3e} > {tol:.1e}"
    return worst


def dev(t, dtype=None):
    t = torch.as_tensor(t)
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def run_prefill(shape, pool, x, g, beta, conv_w, cu, start, init_page, block_table, out_slot,
                raise_on_error=True, max_seq_len=0, workspace=None, path=0):
    """One gdn_prefill_chunked call; returns (o on the host, device error code).
    workspace=False passes none (a tensor-core layer then takes the fused kernel)."""
    T = int(cu[-1])
    o = torch.full((T, shape.num_v_heads, shape.head_dim_v), float("nan"), dtype=shape.torch_out(), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.as_tensor(block_table, dtype=torch.int32)
    if bt.dim() == 1:
        bt = bt[None]
    st = gdn.gdn_prefill_chunked(
        shape, pool, cu_seqlens=dev(cu, torch.int32), start_pos=dev(start, torch.int64),
        init_page=dev(init_page, torch.int32), block_table=dev(bt), out_slot=dev(out_slot, torch.int32),
        x=dev(x), g=dev(g, torch.float32), beta=dev(beta, torch.float32), conv_w=dev(conv_w, torch.float32),
        o=o, dev_error=err, start_pos_host=list(start), init_page_host=list(init_page),
        raise_on_error=raise_on_error, max_seq_len=max_seq_len, workspace=workspace, path=path)
    torch.cuda.synchronize()
    return o.cpu(), int(err.item()), st


def oracle_head(shape, x, g, beta, conv_w, h, cu, start, block_size, S0=None, win0=None):
    """Oracle for one value head only: a 1-qk/1-v-head layer built from the
    channels [q_j | k_j | v_h] that head h reads (j = h // (Hv/Hqk))."""
    G = shape.num_v_heads // shape.num_qk_heads
    j = h // G
    dk, dv, Hqk = shape.head_dim_k, shape.head_dim_v, shape.num_qk_heads
    ch = np.concatenate([np.arange(j * dk, (j + 1) * dk),
                         np.arange(Hqk * dk + j * dk, Hqk * dk + (j + 1) * dk),
                         np.arange(2 * Hqk * dk + h * dv, 2 * Hqk * dk + (h + 1) * dv)])
    xs = x.float().numpy()[:, ch]
    ws = conv_w.float().numpy()[ch]
    d1 = oracle.Dims(1, 1, dk, dv, shape.q_scale, shape.norm_eps)
    S0h = None if S0 is None else np.asarray(S0)[:, h:h + 1]
    w0h = None if win0 is None else np.asarray(win0)[:, :, ch]
    return oracle.prefill(d1, cu, start, block_size, xs, g.float().numpy()[:, h:h + 1],
                          beta.float().numpy()[:, h:h + 1], ws, S0h, w0h)
