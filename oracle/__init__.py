"""CPU oracle for the single-GPU MoE dispatch -> grouped expert MLP -> combine path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It is a thin ctypes wrapper around ``moe_oracle.c`` (plain C, fp64),
which shares no code with the CUDA library and imports nothing from it.

Every function takes and returns numpy arrays.  bf16 values travel as their
raw ``uint16`` bit patterns, FP8 E4M3 codes as ``uint8``, NVFP4 as packed
``uint8`` (two E2M1 codes per byte, the even element in the low nibble) plus
``uint8`` E4M3 block-scale codes.

The page each step follows is cited in ``moe_oracle.c`` beside the step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_BAD_EXPERT = 1
ERR_TOO_MANY_ROUTES = 2

FMT_BF16, FMT_FP8, FMT_NVFP4 = 0, 1, 2
ROUTING_DENSE, ROUTING_SPARSE = 0, 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-D_DEFAULT_SOURCE", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = ctypes.CDLL(_LIB_PATH)
            _lib.moe_oracle_capacity.restype = ctypes.c_int64
            _lib.moe_oracle_capacity.argtypes = [ctypes.c_int64, ctypes.c_double, ctypes.c_int64]
            _lib.moe_oracle_f64_to_bf16.restype = ctypes.c_uint16
            _lib.moe_oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            _lib.moe_oracle_bf16_to_f64.restype = ctypes.c_double
            _lib.moe_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            _lib.moe_oracle_e4m3_to_f64.restype = ctypes.c_double
            _lib.moe_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            _lib.moe_oracle_e2m1_to_f64.restype = ctypes.c_double
            _lib.moe_oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
            _lib.moe_oracle_grouped_mlp_rows.argtypes = (
                [ctypes.c_int] + [ctypes.c_void_p] * 2 + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 7
                + [ctypes.c_double] * 2 + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p])
            _lib.moe_oracle_layer_per_token.argtypes = (
                [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int64] * 3
                + [ctypes.c_void_p] * 2 + [ctypes.c_int64] * 2 + [ctypes.c_void_p] * 6 + [ctypes.c_double] * 2
                + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p])
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 (ties to even), as bit patterns."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().moe_oracle_f64_to_bf16_array(_p(v), ctypes.c_int64(v.size), _p(out))
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    table = np.array([lib.moe_oracle_e4m3_to_f64(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().moe_oracle_f32_to_e4m3_array(_p(v), ctypes.c_int64(v.size), _p(out))
    return out


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    table = np.array([lib.moe_oracle_e2m1_to_f64(c) for c in range(16)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8) & 0xF]


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().moe_oracle_f32_to_e2m1_array(_p(v), ctypes.c_int64(v.size), _p(out))
    return out


def capacity(rows: int, factor: float, align: int = 4) -> int:
    return int(_load().moe_oracle_capacity(int(rows), float(factor), int(align)))


# ----------------------------------------------------------------- the path

def preprocess(fmt: int, routing_map: np.ndarray, T: int, E: int, K: int, m: int, cap: int) -> dict:
    """Counts, padded offsets, row map and overflow flag (see moe_oracle_preprocess)."""
    rmap = _c(routing_map, np.int16 if fmt == ROUTING_DENSE else np.uint8)
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    row_of = np.zeros(T * K, np.int32)
    token_of = np.full(max(cap, 1), -2, np.int32)
    slot_of = np.full(max(cap, 1), -2, np.int32)
    total = np.zeros(1, np.int32)
    ovf = np.zeros(1, np.int32)
    st = _load().moe_oracle_preprocess(
        ctypes.c_int(fmt), _p(rmap), ctypes.c_int64(T), ctypes.c_int64(E), ctypes.c_int64(K),
        ctypes.c_int64(m), ctypes.c_int64(cap), _p(counts), _p(offsets), _p(row_of), _p(token_of),
        _p(slot_of), _p(total), _p(ovf))
    valid = min(int(total[0]), cap)
    return dict(counts=counts, offsets=offsets, row_of=row_of.reshape(T, K), token_of=token_of[:valid],
                slot_of=slot_of[:valid], total_rows=int(total[0]), overflow=int(ovf[0]), status=int(st),
                valid_rows=valid)


def dispatch(fmt: int, routing_map: np.ndarray, probs, pre: dict, x_rows: np.ndarray, cap: int,
             E: int, K: int):
    """Permute rows of ``x_rows`` ([T, ...] any dtype) into a [cap, ...] buffer.

    Returns (Y, Yp); rows at or beyond ``pre['valid_rows']`` are left as zeros here
    and carry no meaning.  Yp is None when ``probs`` is None.
    """
    x = np.ascontiguousarray(x_rows)
    T = x.shape[0]
    row_bytes = x.nbytes // max(T, 1) if T else int(np.prod(x.shape[1:])) * x.itemsize
    y = np.zeros((max(cap, 1),) + x.shape[1:], dtype=x.dtype)
    yp = np.zeros(max(cap, 1), np.float32) if probs is not None else None
    rmap = _c(routing_map, np.int16 if fmt == ROUTING_DENSE else np.uint8)
    pr = _c(probs, np.float32)
    _load().moe_oracle_dispatch(
        ctypes.c_int(fmt), _p(rmap), _p(pr), ctypes.c_int64(T), ctypes.c_int64(E), ctypes.c_int64(K),
        ctypes.c_int64(cap), _p(pre["counts"]), _p(pre["offsets"]),
        _p(np.ascontiguousarray(pre["row_of"], dtype=np.int32)), _p(x), ctypes.c_int64(row_bytes),
        _p(y), _p(yp))
    return y[:cap], (yp[:cap] if yp is not None else None)


def quantize_fp8_rows(x_bf16: np.ndarray):
    """bf16 [T, H] -> (E4M3 codes [T, H], fp32 scales [T, H/128])."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    q = np.empty((T, H), np.uint8)
    s = np.empty((T, H // 128), np.float32)
    _load().moe_oracle_quantize_fp8_rows(_p(x), ctypes.c_int64(T), ctypes.c_int64(H), _p(q), _p(s))
    return q, s


def quantize_fp8_weight(w_bf16: np.ndarray):
    """bf16 [G, N, K] -> (E4M3 codes [G, N, K], fp32 scales [G, N/128, K/128])."""
    w = _c(w_bf16, np.uint16)
    G, N, Kd = w.shape
    q = np.empty((G, N, Kd), np.uint8)
    s = np.empty((G, N // 128, Kd // 128), np.float32)
    _load().moe_oracle_quantize_fp8_weight(_p(w), ctypes.c_int64(G), ctypes.c_int64(N), ctypes.c_int64(Kd),
                                           _p(q), _p(s))
    return q, s


def quantize_nvfp4_rows(x_bf16: np.ndarray, global_scale: float):
    """bf16 [R, K] -> (packed E2M1 [R, K/2], E4M3 block-scale codes [R, K/16])."""
    x = _c(x_bf16, np.uint16)
    shape = x.shape
    x2 = x.reshape(-1, shape[-1])
    R, Kd = x2.shape
    packed = np.empty((R, Kd // 2), np.uint8)
    sc = np.empty((R, Kd // 16), np.uint8)
    _load().moe_oracle_quantize_nvfp4_rows(_p(x2), ctypes.c_int64(R), ctypes.c_int64(Kd),
                                           ctypes.c_float(global_scale), _p(packed), _p(sc))
    return packed.reshape(shape[:-1] + (Kd // 2,)), sc.reshape(shape[:-1] + (Kd // 16,))


def grouped_mlp_rows(fmt: int, y, y_scales, H: int, I: int, E: int, offsets, w13, w13_scales, w2,
                     w2_scales, rows, w13_global=None, w2_global=None, fc1_in_global: float = 0.0,
                     fc2_in_global: float = 0.0, want_act: bool = False, row_probs=None):
    """FFN of the listed permuted rows.  Returns (out bf16 [n, H], act float64 [n, I] or None).
    row_probs ([n]): probabilities applied to the FC2 rows inside the MLP."""
    lib = _load()
    dt = np.uint16 if fmt == FMT_BF16 else np.uint8
    sdt = np.float32 if fmt == FMT_FP8 else np.uint8
    yv, w13v, w2v = _c(y, dt), _c(w13, dt), _c(w2, dt)
    ys = _c(y_scales, sdt) if y_scales is not None else None
    w13s = _c(w13_scales, sdt) if w13_scales is not None else None
    w2s = _c(w2_scales, sdt) if w2_scales is not None else None
    g13 = _c(w13_global, np.float32) if w13_global is not None else None
    g2 = _c(w2_global, np.float32) if w2_global is not None else None
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), H), np.uint16)
    act = np.empty((len(rows), I), np.float64) if want_act else None
    off = _c(offsets, np.int32)
    rp = _c(row_probs, np.float32)
    rc = lib.moe_oracle_grouped_mlp_rows(
        fmt, _p(yv), _p(ys), H, I, E, _p(off), _p(w13v), _p(w13s), _p(g13), _p(w2v), _p(w2s), _p(g2),
        fc1_in_global, fc2_in_global, _p(rows), len(rows), _p(out), _p(act), _p(rp))
    if rc != 0:
        raise ValueError("a listed row lies in no expert segment")
    return out, act


MX_E4M3, MX_E2M1 = 0, 1


def e8m0_decode(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    lib.moe_oracle_e8m0_to_f64.restype = ctypes.c_double
    lib.moe_oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
    table = np.array([lib.moe_oracle_e8m0_to_f64(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def quantize_mx_rows(x_f32: np.ndarray, elem: int):
    """fp32 [R, H] -> (codes: E4M3 [R, H] or packed E2M1 [R, H/2], E8M0 scale codes [R, H/32])."""
    x = _c(x_f32, np.float32)
    R, H = x.shape
    codes = np.empty((R, H if elem == MX_E4M3 else H // 2), np.uint8)
    scales = np.empty((R, H // 32), np.uint8)
    _load().moe_oracle_quantize_mx_rows(_p(x), ctypes.c_int64(R), ctypes.c_int64(H), ctypes.c_int(elem),
                                        _p(codes), _p(scales))
    return codes, scales


def mx_decode_rows(codes: np.ndarray, scales: np.ndarray, elem: int) -> np.ndarray:
    """Decoded float64 values [R, H] of MX rows."""
    codes = np.asarray(codes, np.uint8)
    if elem == MX_E4M3:
        v = e4m3_decode(codes)
    else:
        v = e2m1_decode(np.stack([codes & 0xF, codes >> 4], -1).reshape(codes.shape[0], -1))
    return v * np.repeat(e8m0_decode(scales), 32, axis=1)


def grouped_mlp_rows_mx(fmt: int, y, y_scales, H: int, I: int, E: int, offsets, w13, w13_scales, w2,
                        w2_scales, rows, elem: int, w13_global=None, w2_global=None, fc1_in_global: float = 0.0,
                        fc2_in_global: float = 0.0, row_probs=None):
    """FFN of the listed rows with FC2 written in an MX combine format: (codes, E8M0 scales)."""
    lib = _load()
    dt = np.uint16 if fmt == FMT_BF16 else np.uint8
    sdt = np.float32 if fmt == FMT_FP8 else np.uint8
    yv, w13v, w2v = _c(y, dt), _c(w13, dt), _c(w2, dt)
    ys = _c(y_scales, sdt) if y_scales is not None else None
    w13s = _c(w13_scales, sdt) if w13_scales is not None else None
    w2s = _c(w2_scales, sdt) if w2_scales is not None else None
    g13 = _c(w13_global, np.float32) if w13_global is not None else None
    g2 = _c(w2_global, np.float32) if w2_global is not None else None
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    codes = np.empty((len(rows), H if elem == MX_E4M3 else H // 2), np.uint8)
    scales = np.empty((len(rows), H // 32), np.uint8)
    off = _c(offsets, np.int32)
    fn = lib.moe_oracle_grouped_mlp_rows_mx
    fn.argtypes = ([ctypes.c_int] + [ctypes.c_void_p] * 2 + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 7
                   + [ctypes.c_double] * 2 + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p])
    rp = _c(row_probs, np.float32)
    rc = fn(fmt, _p(yv), _p(ys), H, I, E, _p(off), _p(w13v), _p(w13s), _p(g13), _p(w2v), _p(w2s), _p(g2),
            fc1_in_global, fc2_in_global, _p(rows), len(rows), elem, _p(codes), _p(scales), _p(rp))
    if rc != 0:
        raise ValueError("a listed row lies in no expert segment")
    return codes, scales


def combine_mx(codes: np.ndarray, scales: np.ndarray, elem: int, row_of: np.ndarray, perm_probs=None):
    """y[t] = bf16(sum_k w * decoded O[row_of[t, k]]) from MX expert rows."""
    c = _c(codes, np.uint8)
    sc = _c(scales, np.uint8)
    ro = _c(row_of, np.int32)
    T, K = ro.shape
    H = sc.shape[1] * 32
    pp = _c(perm_probs, np.float32)
    y = np.empty((T, H), np.uint16)
    _load().moe_oracle_combine_mx(_p(c), _p(sc), ctypes.c_int64(H), ctypes.c_int(elem), _p(ro), ctypes.c_int64(T),
                                  ctypes.c_int64(K), _p(pp), _p(y))
    return y


def combine(o_bf16: np.ndarray, row_of: np.ndarray, perm_probs=None) -> np.ndarray:
    """y[t] = bf16(sum_k w * O[row_of[t, k]]) over kept routes."""
    o = _c(o_bf16, np.uint16)
    ro = _c(row_of, np.int32)
    T, K = ro.shape
    H = o.shape[1]
    pp = _c(perm_probs, np.float32)
    y = np.empty((T, H), np.uint16)
    _load().moe_oracle_combine(_p(o), ctypes.c_int64(H), _p(ro), ctypes.c_int64(T), ctypes.c_int64(K),
                               _p(pp), _p(y))
    return y


def combine_backward(g_y: np.ndarray, pre: dict, cap: int, o=None, perm_probs=None):
    """Backward of combine: (gO bf16 [cap, H], gw fp32 [cap] or None).  gw is
    formed when both ``o`` and ``perm_probs`` are given.  Rows at or beyond
    ``pre['valid_rows']`` are zeros here and carry no meaning."""
    gy = _c(g_y, np.uint16)
    T, H = gy.shape
    ro = np.ascontiguousarray(pre["row_of"], dtype=np.int32)
    K = ro.shape[1]
    E = len(pre["counts"])
    ov = _c(o, np.uint16) if o is not None else None
    pp = _c(perm_probs, np.float32)
    g_o = np.zeros((max(cap, 1), H), np.uint16)
    g_w = np.zeros(max(cap, 1), np.float32) if (o is not None and perm_probs is not None) else None
    _load().moe_oracle_combine_backward(
        _p(gy), ctypes.c_int64(T), ctypes.c_int64(H), ctypes.c_int64(E), ctypes.c_int64(K), _p(ro),
        _p(pre["counts"]), _p(pre["offsets"]), ctypes.c_int64(cap), _p(ov), _p(pp), _p(g_o), _p(g_w))
    return g_o[:cap], (g_w[:cap] if g_w is not None else None)


def dispatch_backward(fmt: int, routing_map, row_of, E: int, g_y, g_yp=None):
    """Backward of dispatch: (gx bf16 [T, H], gp fp32 in the routing layout or None)."""
    rmap = _c(routing_map, np.int16 if fmt == ROUTING_DENSE else np.uint8)
    ro = np.ascontiguousarray(row_of, dtype=np.int32)
    T, K = ro.shape
    gy = _c(g_y, np.uint16)
    H = gy.shape[1]
    gyp = _c(g_yp, np.float32)
    g_x = np.empty((T, H), np.uint16)
    g_p = None
    if g_yp is not None:
        g_p = np.empty((T, K) if fmt == ROUTING_DENSE else (T, E), np.float32)
    _load().moe_oracle_dispatch_backward(
        ctypes.c_int(fmt), _p(rmap), ctypes.c_int64(T), ctypes.c_int64(E), ctypes.c_int64(K), ctypes.c_int64(H),
        _p(ro), _p(gy), _p(gyp), _p(g_x), _p(g_p))
    return g_x, g_p


def layer_per_token(fmt: int, routing_fmt: int, routing_map, probs, E: int, K: int, x, x_scales, H: int,
                    I: int, w13, w13_scales, w2, w2_scales, tokens, w13_global=None, w2_global=None,
                    fc1_in_global: float = 0.0, fc2_in_global: float = 0.0) -> np.ndarray:
    """The whole layer per token, without permutation (independent formulation)."""
    lib = _load()
    dt = np.uint16 if fmt == FMT_BF16 else np.uint8
    sdt = np.float32 if fmt == FMT_FP8 else np.uint8
    rmap = _c(routing_map, np.int16 if routing_fmt == ROUTING_DENSE else np.uint8)
    T = rmap.shape[0]
    pr = _c(probs, np.float32)
    xv = _c(x, dt)
    xs = _c(x_scales, sdt) if x_scales is not None else None
    w13v, w2v = _c(w13, dt), _c(w2, dt)
    w13s = _c(w13_scales, sdt) if w13_scales is not None else None
    w2s = _c(w2_scales, sdt) if w2_scales is not None else None
    g13 = _c(w13_global, np.float32) if w13_global is not None else None
    g2 = _c(w2_global, np.float32) if w2_global is not None else None
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    y = np.empty((len(tokens), H), np.uint16)
    lib.moe_oracle_layer_per_token(fmt, routing_fmt, _p(rmap), _p(pr), T, E, K, _p(xv), _p(xs), H, I,
                                   _p(w13v), _p(w13s), _p(g13), _p(w2v), _p(w2s), _p(g2), fc1_in_global,
                                   fc2_in_global, _p(tokens), len(tokens), _p(y))
    return y
