"""CPU oracle of the MoE expert step -- TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper over `oracle.cpp` (plain scalar C++).  Only the tests,
the smoke check and the benchmark's timed CPU-baseline leg may import this
package; the product library never does.  It shares no code with the CUDA
path.  See `oracle.cpp` for the page citations of each function.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (plain g++, no fast-math; with
    OpenMP for the optional multi-threaded row loops when the compiler has it)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        base = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared"]
        try:
            subprocess.check_call(base + ["-fopenmp", "-o", tmp, _SRC],
                                  stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base + ["-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _p(a, ct):
    return a.ctypes.data_as(C.POINTER(ct))


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        i32, i64, f32, vp = C.c_int, C.c_int64, C.c_float, C.c_void_p
        L.or_expert_bytes.restype = i64
        L.or_expert_bytes.argtypes = [i32, i32]
        L.or_blob_offsets.argtypes = [i32, i32, vp]
        L.or_dequant.argtypes = [vp, vp, vp, i32, i32, vp]
        L.or_blob_matrix.argtypes = [vp, i32, i32, i32, vp]
        L.or_exp.restype = f32
        L.or_exp.argtypes = [f32]
        L.or_sigmoid.restype = f32
        L.or_sigmoid.argtypes = [f32]
        L.or_router_logits.restype = i32
        L.or_router_logits.argtypes = [vp, vp, i32, i32, i32, vp]
        L.or_route_softmax_topk.restype = i32
        L.or_route_softmax_topk.argtypes = [vp, i32, i32, i32, vp, vp]
        L.or_route_sigmoid_group.restype = i32
        L.or_route_sigmoid_group.argtypes = [vp, vp, i32, i32, i32, i32, i32, f32, vp, vp]
        L.or_q_star.restype = i32
        L.or_q_star.argtypes = [i32, i32, i32]
        L.or_cache_step.restype = i32
        L.or_cache_step.argtypes = [i32, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                    vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.or_cache_place.restype = i32
        L.or_cache_place.argtypes = [i32, i32, i32, i32, vp, i32, vp, vp, vp, vp]
        L.or_slots_for_budget.restype = i64
        L.or_slots_for_budget.argtypes = [i64, i64]
        L.or_cache_resize.restype = i32
        L.or_cache_resize.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.or_expert_forward.argtypes = [vp, i32, i32, vp, i32, vp]
        f64 = C.c_double
        for name in ("or_e2m1", "or_e4m3", "or_e8m0"):
            getattr(L, name).restype = f64
            getattr(L, name).argtypes = [i32]
        L.or_fp4_blob_offsets.restype = i32
        L.or_fp4_blob_offsets.argtypes = [i32, i32, i32, vp]
        L.or_fp4_blob_matrix.restype = i32
        L.or_fp4_blob_matrix.argtypes = [vp, i32, i32, i32, i32, vp]
        L.or_fp4_expert_forward.restype = i32
        L.or_fp4_expert_forward.argtypes = [vp, i32, i32, i32, vp, i32, vp]
        L.or_moe_ffn.argtypes = [vp, i32, i32, i32, vp, i32, vp, vp, i32, vp, i32, vp]
        L.or_set_threads.restype = i32
        L.or_set_threads.argtypes = [i32]
        _lib = L
    return _lib


def _vp(a):
    return C.c_void_p(a.ctypes.data) if a is not None else None


# --------------------------------------------------------------- wrappers
def expert_bytes(H: int, I: int) -> int:
    return int(lib().or_expert_bytes(H, I))


def blob_offsets(H: int, I: int) -> dict:
    off = np.zeros(10, dtype=np.int64)
    lib().or_blob_offsets(H, I, _vp(off))
    names = ("gq", "uq", "dq", "gs", "gb", "us", "ub", "ds", "db", "total")
    return {n: int(v) for n, v in zip(names, off)}


def dequant(codes: np.ndarray, s: np.ndarray, b: np.ndarray, rows: int, cols: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().or_dequant(_vp(codes), _vp(s), _vp(b), rows, cols, _vp(out))
    return out


def blob_matrix(blob: np.ndarray, H: int, I: int, which: int) -> np.ndarray:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    shape = (I, H) if which in (0, 1) else (H, I)
    out = np.empty(shape, dtype=np.float32)
    lib().or_blob_matrix(_vp(blob), H, I, which, _vp(out))
    return out


def exp(x: float) -> float:
    return float(lib().or_exp(float(x)))


def sigmoid(z: float) -> float:
    return float(lib().or_sigmoid(float(z)))


def router_logits(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    T, H = x.shape
    E = w.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    rc = lib().or_router_logits(_vp(x), _vp(w), T, E, H, _vp(out))
    if rc:
        raise ValueError("router_logits: bad shape")
    return out


def route_softmax_topk(logits: np.ndarray, k: int):
    l = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = l.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    if lib().or_route_softmax_topk(_vp(l), T, E, k, _vp(ids), _vp(w)):
        raise ValueError("route_softmax_topk: bad arguments")
    return ids, w


def route_sigmoid_group(logits, bias, n_groups, topk_groups, k, scale):
    l = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = l.shape
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    if lib().or_route_sigmoid_group(_vp(l), _vp(bias), T, E, n_groups, topk_groups, k,
                                    float(scale), _vp(ids), _vp(w)):
        raise ValueError("route_sigmoid_group: bad arguments")
    return ids, w


def q_star(m: int, bp: int, bh: int) -> int:
    return int(lib().or_q_star(m, bp, bh))


class CacheState:
    """Host copy of the slot cache tables for the oracle control step."""

    def __init__(self, n_ids: int, S: int):
        self.slot_of_id = np.full(n_ids, -1, dtype=np.int32)
        self.id_of_slot = np.full(S, -1, dtype=np.int32)
        self.ts = np.zeros(S, dtype=np.uint32)
        self.clock = np.zeros(1, dtype=np.uint32)

    def copy(self):
        c = CacheState.__new__(CacheState)
        c.slot_of_id = self.slot_of_id.copy()
        c.id_of_slot = self.id_of_slot.copy()
        c.ts = self.ts.copy()
        c.clock = self.clock.copy()
        return c


SHARED_LRU, LAYER_LRU, STATIC = 0, 1, 2


def cache_place(state: CacheState, E: int, L: int, ids, policy: int = SHARED_LRU):
    """Empty `state`, then preload the bank ids `ids` (l*E + e) into slots."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    rc = lib().or_cache_place(E, L, state.id_of_slot.size, policy, _vp(ids), ids.size,
                              _vp(state.slot_of_id), _vp(state.id_of_slot), _vp(state.ts),
                              _vp(state.clock))
    if rc:
        raise ValueError("cache_place: bad id list for this cache / policy")


def cache_step(state: CacheState, E: int, layer: int, ids: np.ndarray, K: int, bp: int, bh: int,
               policy: int = SHARED_LRU, L: int = 1):
    """Run one control step in place on `state`; return the plan as a dict.
    `L` (the number of layers) matters only for the per-layer policy."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    n = ids.size
    S = state.id_of_slot.size
    cap = max(n, 1)
    bufs = {k: np.full(cap, -1, dtype=np.int32) for k in
            ("uniq", "hit_ids", "hit_slots", "fill_ids", "fill_slots", "evicted_ids", "direct_ids")}
    victims = np.full(max(K, 1), -1, dtype=np.int32)
    counts = np.zeros(8, dtype=np.int32)
    rc = lib().or_cache_step(E, layer, _vp(ids), n, S, K, bp, bh, policy, L,
                             _vp(state.slot_of_id), _vp(state.id_of_slot), _vp(state.ts),
                             _vp(state.clock), _vp(bufs["uniq"]), _vp(bufs["hit_ids"]),
                             _vp(bufs["hit_slots"]), _vp(bufs["fill_ids"]), _vp(bufs["fill_slots"]),
                             _vp(bufs["evicted_ids"]), _vp(bufs["direct_ids"]), _vp(victims),
                             _vp(counts))
    if rc:
        raise ValueError("cache_step: routed id out of range or bad policy")
    n_uniq, n_hit, n_miss, q, n_fill, n_direct, n_vict, now = (int(v) for v in counts)
    return {
        "uniq": bufs["uniq"][:n_uniq].copy(),
        "hit_ids": bufs["hit_ids"][:n_hit].copy(),
        "hit_slots": bufs["hit_slots"][:n_hit].copy(),
        "fill_ids": bufs["fill_ids"][:n_fill].copy(),
        "fill_slots": bufs["fill_slots"][:n_fill].copy(),
        "evicted_ids": bufs["evicted_ids"][:n_fill].copy(),
        "direct_ids": bufs["direct_ids"][:n_direct].copy(),
        "victims": victims[:K].copy(),
        "counts": counts.copy(),
        "n_uniq": n_uniq, "n_hit": n_hit, "n_miss": n_miss, "q": q, "n_fill": n_fill,
        "n_direct": n_direct, "n_victims": n_vict, "now": now,
    }


def slots_for_budget(free_bytes: int, slot_bytes: int) -> int:
    """floor(free_bytes / slot_bytes): the slots a memory budget holds."""
    n = int(lib().or_slots_for_budget(int(free_bytes), int(slot_bytes)))
    if n < 0:
        raise ValueError("slots_for_budget: bad sizes")
    return n


def cache_resize(state: CacheState, S_new: int) -> dict:
    """Re-divide the slot pool of `state` into S_new slots (in place: the slot
    arrays are replaced by arrays of S_new entries).  Returns the evicted ids,
    the (from, to) blob moves and the counts."""
    S = state.id_of_slot.size
    cap = max(S, S_new)
    ios = np.full(cap, -1, dtype=np.int32)
    ios[:S] = state.id_of_slot
    ts = np.zeros(cap, dtype=np.uint32)
    ts[:S] = state.ts
    ev = np.full(cap, -1, dtype=np.int32)
    mf = np.full(cap, -1, dtype=np.int32)
    mt = np.full(cap, -1, dtype=np.int32)
    counts = np.zeros(3, dtype=np.int32)
    rc = lib().or_cache_resize(state.slot_of_id.size, S, S_new, _vp(state.slot_of_id), _vp(ios),
                               _vp(ts), _vp(ev), _vp(mf), _vp(mt), _vp(counts))
    if rc:
        raise ValueError("cache_resize: bad sizes or tables")
    n_ev, n_mv, n_occ = (int(v) for v in counts)
    state.id_of_slot = ios[:S_new].copy()
    state.ts = ts[:S_new].copy()
    return {"evicted_ids": ev[:n_ev].copy(), "move_from": mf[:n_mv].copy(),
            "move_to": mt[:n_mv].copy(), "n_evicted": n_ev, "n_moved": n_mv, "n_occupied": n_occ}


def expert_forward(blob: np.ndarray, H: int, I: int, x_bits: np.ndarray) -> np.ndarray:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1, H)
    y = np.empty((x.shape[0], H), dtype=np.float64)
    lib().or_expert_forward(_vp(blob), H, I, _vp(x), x.shape[0], _vp(y))
    return y


def moe_ffn(blobs, H: int, I: int, x_bits: np.ndarray, ids: np.ndarray, wts: np.ndarray,
            shared_blob=None, shared_I: int = 0) -> np.ndarray:
    """Layer output y[T][H] (float64).  blobs: sequence of E uint8 blobs (or a 2-D array)."""
    blobs = [np.ascontiguousarray(b, dtype=np.uint8) for b in blobs]
    E = len(blobs)
    ptrs = (C.c_void_p * E)(*[b.ctypes.data for b in blobs])
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1, H)
    T = x.shape[0]
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(T, -1)
    wts = np.ascontiguousarray(wts, dtype=np.float32).reshape(T, -1)
    k = ids.shape[1]
    assert ids.min(initial=0) >= 0 and ids.max(initial=0) < E
    sb = None if shared_blob is None else np.ascontiguousarray(shared_blob, dtype=np.uint8)
    y = np.empty((T, H), dtype=np.float64)
    lib().or_moe_ffn(C.cast(ptrs, C.c_void_p), E, H, I, _vp(x), T, _vp(ids), _vp(wts), k,
                     _vp(sb), shared_I, _vp(y))
    return y


# ------------------------------------------------------ FP4 expert formats
MXFP4, NVFP4 = 0, 1


def e2m1(code: int) -> float:
    return float(lib().or_e2m1(int(code)))


def e4m3(byte: int) -> float:
    return float(lib().or_e4m3(int(byte)))


def e8m0(byte: int) -> float:
    return float(lib().or_e8m0(int(byte)))


def fp4_blob_offsets(H: int, I: int, fmt: int) -> dict:
    off = np.zeros(8, dtype=np.int64)
    if lib().or_fp4_blob_offsets(H, I, fmt, _vp(off)):
        raise ValueError("fp4_blob_offsets: bad format or shape")
    keys = ("gq", "uq", "dq", "gs", "us", "ds", "mat", "total")
    return {k: int(v) for k, v in zip(keys, off)}


def fp4_blob_matrix(blob: np.ndarray, H: int, I: int, which: int, fmt: int) -> np.ndarray:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    rows, cols = (H, I) if which == 2 else (I, H)
    out = np.empty((rows, cols), dtype=np.float64)
    if lib().or_fp4_blob_matrix(_vp(blob), H, I, which, fmt, _vp(out)):
        raise ValueError("fp4_blob_matrix: bad arguments")
    return out


def fp4_expert_forward(blob: np.ndarray, H: int, I: int, fmt: int, x_bits: np.ndarray) -> np.ndarray:
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1, H)
    y = np.empty(x_bits.shape, dtype=np.float64)
    if lib().or_fp4_expert_forward(_vp(blob), H, I, fmt, _vp(x_bits), x_bits.shape[0], _vp(y)):
        raise ValueError("fp4_expert_forward: bad arguments")
    return y


def set_threads(n: int) -> int:
    """Host threads for the oracle's row loops (dequantisation, float64 expert);
    returns the count in effect (1 without OpenMP).  Results do not depend on it."""
    return int(lib().or_set_threads(int(n)))
