"""fp64 CPU oracle of the Gated DeltaNet state path.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  It shares no code with the CUDA engine; both sides only share the
seeded input generators (``gated_deltanet_state_gb300.inputs``), which hold
none of the method's arithmetic.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision, token by
token).  This module builds and loads it, widens inputs to float64 exactly as
the GPU receives them, and composes the replay operations out of the same
recurrence:

* ``prefill``   — conv + SiLU, L2 norm, gated delta rule, block checkpoints
  ("Prefix caching on Gated DeltaNet hybrids", "Why hits were wrong";
  "Hybrid linear attention (gated DeltaNet)", "Why this family is different").
* ``decode``    — the same step for one token per sequence.
* ``replay_append`` / ``replay_rollback`` / ``replay_flush`` — one checkpoint
  plus a log of inputs since it; outputs come from the two, rollback drops
  log rows, the flush rewrites the checkpoint ("Caching less to serve more
  requests", "What we changed").
* ``core_prefill`` / ``core_decode`` — the packed core: gates from the b | a
  rows, the same recurrence, gated RMS norm of the outputs ("Hybrid linear
  attention (gated DeltaNet)", "Packed-core traces").

Every function is pinned in ``tests/test_oracle_pins.py`` against brute force,
closed forms, identities and the pages' worked values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

CONV_K = 4


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/liboracle.so with gcc (no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.gdn_oracle_prefill.argtypes = [ctypes.c_int] * 4 + [f64, f64, i32, P, P, i64] + [P] * 10 + [ctypes.c_int]
        lib.gdn_oracle_prefill.restype = ctypes.c_int
        lib.gdn_oracle_recurrence.argtypes = [ctypes.c_int, ctypes.c_int, i64] + [P] * 7
        lib.gdn_oracle_recurrence.restype = ctypes.c_int
        lib.gdn_oracle_conv_silu.argtypes = [i64, i64, P, P, P, P]
        lib.gdn_oracle_conv_silu.restype = ctypes.c_int
        lib.gdn_oracle_l2norm.argtypes = [ctypes.c_int, P, f64, f64]
        lib.gdn_oracle_l2norm.restype = ctypes.c_int
        lib.gdn_oracle_num_threads.argtypes = []
        lib.gdn_oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().gdn_oracle_num_threads())


def _f64(a) -> np.ndarray:
    """Exact widening to a C-contiguous float64 array (torch or numpy input)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Dims:
    """Layer shape: qk heads, v heads, head dims, q scale and norm epsilon."""
    Hqk: int
    Hv: int
    dk: int
    dv: int
    q_scale: float = 1.0
    eps: float = 1e-6

    @property
    def conv_dim(self) -> int:
        return 2 * self.Hqk * self.dk + self.Hv * self.dv


def conv_silu(x, win, conv_w) -> np.ndarray:
    """SiLU(causal depthwise conv, kernel 4) over all channels: [T][conv_dim]."""
    x, win, w = _f64(x), _f64(win), _f64(conv_w)
    T, cd = x.shape
    y = np.empty((T, cd), np.float64)
    _load().gdn_oracle_conv_silu(cd, T, _p(x), _p(win), _p(w), _p(y))
    return y


def l2norm(v, scale: float = 1.0, eps: float = 1e-6) -> np.ndarray:
    v = _f64(v).copy()
    _load().gdn_oracle_l2norm(v.size, _p(v), float(scale), float(eps))
    return v


def recurrence(q, k, v, a, b, S0):
    """Bare gated delta rule for one head: returns (S_T, o [T][dv])."""
    q, k, v, a, b = _f64(q), _f64(k), _f64(v), _f64(a), _f64(b)
    S = _f64(S0).copy()
    T, dk = k.shape
    dv = v.shape[1]
    o = np.empty((T, dv), np.float64)
    _load().gdn_oracle_recurrence(dk, dv, T, _p(q), _p(k), _p(v), _p(a), _p(b), _p(S), _p(o))
    return S, o


def boundaries(start_pos: int, n_tokens: int, block_size: int) -> list[int]:
    """Absolute positions P = j*B with start_pos < P <= start_pos + n_tokens."""
    first = start_pos // block_size + 1
    last = (start_pos + n_tokens) // block_size
    return [j * block_size for j in range(first, last + 1)]


def prefill(d: Dims, cu_seqlens, start_pos, block_size: int, x, g, beta, conv_w,
            S0=None, win0=None, nthreads: int = 0):
    """Run the oracle prefill.

    Returns a dict with o [T][Hv][dv], S [N][Hv][dv][dk] (final), win
    [N][3][conv_dim] (final), ck_S / ck_win (one entry per crossed boundary,
    sequences in order) and ck_off [N+1].
    """
    cu = _i64(cu_seqlens)
    sp = _i64(start_pos)
    N = len(cu) - 1
    x, g, beta, w = _f64(x), _f64(g), _f64(beta), _f64(conv_w)
    T = int(cu[-1])
    assert x.shape == (T, d.conv_dim), (x.shape, T, d.conv_dim)
    S = (np.zeros((N, d.Hv, d.dv, d.dk)) if S0 is None else _f64(S0).reshape(N, d.Hv, d.dv, d.dk).copy())
    win = (np.zeros((N, CONV_K - 1, d.conv_dim)) if win0 is None
           else _f64(win0).reshape(N, CONV_K - 1, d.conv_dim).copy())
    counts = [len(boundaries(int(sp[s]), int(cu[s + 1] - cu[s]), block_size)) for s in range(N)]
    ck_off = np.zeros(N + 1, np.int64)
    ck_off[1:] = np.cumsum(counts)
    nck = int(ck_off[-1])
    ck_S = np.zeros((max(nck, 1), d.Hv, d.dv, d.dk))
    ck_win = np.zeros((max(nck, 1), CONV_K - 1, d.conv_dim))
    o = np.zeros((T, d.Hv, d.dv))
    rc = _load().gdn_oracle_prefill(d.Hqk, d.Hv, d.dk, d.dv, float(d.q_scale), float(d.eps), N,
                                    _p(cu), _p(sp), int(block_size), _p(x), _p(g), _p(beta), _p(w),
                                    _p(S), _p(win), _p(o), _p(ck_off), _p(ck_S), _p(ck_win),
                                    int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle prefill failed ({rc})")
    return {"o": o, "S": S, "win": win, "ck_S": ck_S[:nck], "ck_win": ck_win[:nck], "ck_off": ck_off}


def decode(d: Dims, x, g, beta, conv_w, S0, win0, nthreads: int = 0):
    """One token per sequence from (S0, win0): returns (o [N][Hv][dv], S, win)."""
    x = _f64(x)
    N = x.shape[0]
    cu = np.arange(N + 1, dtype=np.int64)
    # Block size beyond any position: a decode step writes no checkpoint.
    r = prefill(d, cu, np.zeros(N, np.int64), 1 << 62, x, g, beta, conv_w, S0, win0, nthreads)
    return r["o"], r["S"], r["win"]


def replay_append(d: Dims, conv_w, S_ckpt, win_ckpt, log_x, log_g, log_b, log_len,
                  x_new, g_new, b_new, nthreads: int = 0):
    """Outputs of the new rows, computed from the checkpoint and the log.

    Request r runs the recurrence from (S_ckpt[r], win_ckpt[r]) over its
    log_len[r] logged rows and then the m new rows; the outputs of the new rows
    are returned as [N][m][Hv][dv].  The checkpoint is not changed.
    """
    log_x, log_g, log_b = _f64(log_x), _f64(log_g), _f64(log_b)
    x_new, g_new, b_new = _f64(x_new), _f64(g_new), _f64(b_new)
    lens = _i64(log_len)
    N, m = x_new.shape[0], x_new.shape[1]
    xs, gs, bs, cu = [], [], [], [0]
    for r in range(N):
        n = int(lens[r])
        xs += [log_x[r, :n], x_new[r]]
        gs += [log_g[r, :n], g_new[r]]
        bs += [log_b[r, :n], b_new[r]]
        cu.append(cu[-1] + n + m)
    res = prefill(d, np.array(cu), np.zeros(N, np.int64), 1 << 62, np.concatenate(xs),
                  np.concatenate(gs), np.concatenate(bs), conv_w, S_ckpt, win_ckpt, nthreads)
    o = np.stack([res["o"][cu[r + 1] - m:cu[r + 1]] for r in range(N)])
    return o


def replay_rollback(log_len, accepted, num_appended: int) -> np.ndarray:
    """Drop the rejected rows of the last append: len - (appended - accepted)."""
    lens, acc = _i64(log_len), _i64(accepted)
    assert np.all((acc >= 0) & (acc <= num_appended))
    return lens - (num_appended - acc)


def replay_flush(d: Dims, conv_w, S_ckpt, win_ckpt, log_x, log_g, log_b, log_len, nthreads: int = 0):
    """Apply the kept log rows to the checkpoint: returns (S, win) after them."""
    log_x, log_g, log_b = _f64(log_x), _f64(log_g), _f64(log_b)
    lens = _i64(log_len)
    N = log_x.shape[0]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    xs = np.concatenate([log_x[r, :lens[r]] for r in range(N)]) if cu[-1] else np.zeros((0, d.conv_dim))
    gs = np.concatenate([log_g[r, :lens[r]] for r in range(N)]) if cu[-1] else np.zeros((0, d.Hv))
    bs = np.concatenate([log_b[r, :lens[r]] for r in range(N)]) if cu[-1] else np.zeros((0, d.Hv))
    res = prefill(d, cu, np.zeros(N, np.int64), 1 << 62, xs, gs, bs, conv_w, S_ckpt, win_ckpt, nthreads)
    return res["S"], res["win"]


# --------------------------------------------------------------------------- packed core
# "Hybrid linear attention (gated DeltaNet)", "Packed-core traces": the core
# takes packed qkvz plus ba per token and returns gated-normalised value rows;
# it owns the conv weights, dt_bias, a float32 A_log and the norm scale.  The
# pages name the weights only; the gates and the norm are read as
#   g    = -exp(A_log) * softplus(a + dt_bias)      (so a_t = exp(g))
#   beta = sigmoid(b)
#   y    = o / sqrt(mean_dv(o^2) + eps) * norm_w * silu(z)   per token and v head.


def softplus(x) -> np.ndarray:
    """log(1 + e^x), evaluated as max(x, 0) + log1p(e^-|x|)."""
    x = _f64(x)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def core_gates(ba, A_log, dt_bias, Hv: int):
    """Gates from the packed b | a rows [T][2 Hv]: (g, beta), each [T][Hv]."""
    ba = _f64(ba).reshape(-1, 2 * Hv)
    b, a = ba[:, :Hv], ba[:, Hv:]
    g = -np.exp(_f64(A_log))[None, :] * softplus(a + _f64(dt_bias)[None, :])
    beta = 1.0 / (1.0 + np.exp(-b))
    return g, beta


def gated_rmsnorm(o, z, norm_w, eps: float):
    """RMS-normalise o [..., dv] over dv, scale by norm_w [dv], gate by silu(z)."""
    o, z, w = _f64(o), _f64(z), _f64(norm_w)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o / rms * w * (z / (1.0 + np.exp(-z)))


def _split_qkvz(d: Dims, qkvz):
    qkvz = _f64(qkvz)
    return qkvz[:, :d.conv_dim], qkvz[:, d.conv_dim:].reshape(-1, d.Hv, d.dv)


def core_prefill(d: Dims, cu_seqlens, start_pos, block_size: int, qkvz, ba, conv_w, A_log, dt_bias,
                 norm_w, norm_eps: float, S0=None, win0=None, nthreads: int = 0):
    """The prefill from packed inputs: gates from ba, the recurrence on the
    q | k | v part, the gated norm on its outputs (returned as "y"; the rest
    as ``prefill`` returns it)."""
    x, z = _split_qkvz(d, qkvz)
    g, beta = core_gates(ba, A_log, dt_bias, d.Hv)
    r = prefill(d, cu_seqlens, start_pos, block_size, x, g, beta, conv_w, S0, win0, nthreads)
    r["y"] = gated_rmsnorm(r["o"], z, norm_w, norm_eps)
    return r


def core_decode(d: Dims, qkvz, ba, conv_w, A_log, dt_bias, norm_w, norm_eps: float, S0, win0,
                nthreads: int = 0):
    """One packed token per sequence: returns (y [N][Hv][dv], S, win)."""
    x, z = _split_qkvz(d, qkvz)
    g, beta = core_gates(ba, A_log, dt_bias, d.Hv)
    o, S, win = decode(d, x, g, beta, conv_w, S0, win0, nthreads)
    return gated_rmsnorm(o, z, norm_w, norm_eps), S, win
