"""Python binding of libmoe.so, the GB300-native MoE expert step.

The functions below carry the C entry points' names and only marshal
arguments (device pointers, sizes, the CUDA stream) into ctypes calls; every
step of the computation runs in the library's CUDA kernels.  PyTorch is used
by the helper classes for device memory and streams only.

The library must be built first (``__graft_entry__.build()`` or
``python -m moe_expert_offload_gb300._build``); importing the binding without
it raises, there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

from . import _build

MOE_OK = 0
MOE_EINVAL = -1
MOE_ECUDA = -2
MOE_EUNSUPPORTED = -3
MOE_ECAPACITY = -4
MOE_ETIMEOUT = -5
MOE_ROUTER_SOFTMAX_TOPK = 0
MOE_ROUTER_SIGMOID_GROUP = 1
MOE_DERR_BAD_ID = 1
MOE_DERR_WAIT = 2
MOE_DERR_RANGE = 4  # checked builds only (libmoe_checked.so)

EXPORTED = (
    "moe_last_error", "moe_version", "moe_expert_bytes", "moe_route", "moe_cache_reset",
    "moe_cache_step", "moe_ffn_workspace_bytes", "moe_expert_ffn", "moe_layer_workspace_bytes",
    "moe_layer_forward", "moe_expert_ffn_noalloc", "moe_prefill_workspace_bytes",
    "moe_layer_prefetch", "moe_expert_ffn_prefill", "moe_layer_forward_prefill",
    "moe_slots_for_budget", "moe_cache_resize_workspace_bytes", "moe_cache_resize",
)
MOE_NOALLOC_SCRATCH_BYTES = 8 << 20


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class MoeSpec(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("hidden", C.c_int32), ("inter", C.c_int32),
                ("num_experts", C.c_int32), ("top_k", C.c_int32), ("router", C.c_int32),
                ("n_groups", C.c_int32), ("topk_groups", C.c_int32), ("routed_scale", C.c_float),
                ("group_size", C.c_int32), ("has_shared", C.c_int32),
                ("shared_inter", C.c_int32), ("format", C.c_int32)]


# moe_spec.format values (include/moe.h)
FORMAT_INT4, FORMAT_MXFP4, FORMAT_NVFP4 = 0, 1, 2


class MoeCache(C.Structure):
    _fields_ = [("num_slots", C.c_int32), ("k_victims", C.c_int32), ("bp_mbps", C.c_int32),
                ("bh_mbps", C.c_int32), ("slot_of_id", C.c_void_p), ("id_of_slot", C.c_void_p),
                ("ts", C.c_void_p), ("clock", C.c_void_p), ("slot_pool", C.c_void_p),
                ("bank", C.c_void_p), ("policy", C.c_int32), ("sync", C.c_void_p)]


# words behind moe_cache.sync (include/moe.h)
CACHE_SYNC_WORDS = 4096


# moe_cache.policy values (include/moe.h)
POLICY_SHARED_LRU, POLICY_LAYER_LRU, POLICY_STATIC = 0, 1, 2


class MoePlan(C.Structure):
    _fields_ = [("capacity", C.c_int32), ("uniq", C.c_void_p), ("hit_ids", C.c_void_p),
                ("hit_slots", C.c_void_p), ("fill_ids", C.c_void_p), ("fill_slots", C.c_void_p),
                ("evicted_ids", C.c_void_p), ("direct_ids", C.c_void_p), ("victims", C.c_void_p),
                ("counts", C.c_void_p), ("err", C.c_void_p)]


_lib = None


def library_path() -> str:
    """libmoe.so, or the library named by MOE_LIBRARY (e.g. the checked build,
    libmoe_checked.so)."""
    return os.environ.get("MOE_LIBRARY") or _build.LIB


def lib():
    """Load libmoe.so; raise if it has not been built (no fallback path exists)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{os.path.basename(path)} is not built; run "
                               "__graft_entry__.build() first")
        L = C.CDLL(path)
        vp, i32, sz = C.c_void_p, C.c_int32, C.c_size_t
        sp, cp, pp = C.POINTER(MoeSpec), C.POINTER(MoeCache), C.POINTER(MoePlan)
        L.moe_last_error.restype = C.c_char_p
        L.moe_version.restype = C.c_char_p
        L.moe_expert_bytes.restype = sz
        L.moe_expert_bytes.argtypes = [sp]
        L.moe_route.restype = C.c_int
        L.moe_route.argtypes = [sp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_cache_reset.restype = C.c_int
        L.moe_cache_reset.argtypes = [sp, cp, vp]
        L.moe_debug_inject_ffn_stall.restype = C.c_int
        L.moe_debug_inject_ffn_stall.argtypes = [i32]
        L.moe_layer_kernel_count.restype = i32
        L.moe_layer_kernel_count.argtypes = [sp, cp, i32]
        L.moe_cache_place.restype = C.c_int
        L.moe_cache_place.argtypes = [sp, cp, vp, i32, vp]
        L.moe_slots_for_budget.restype = C.c_int64
        L.moe_slots_for_budget.argtypes = [sp, C.c_int64]
        L.moe_cache_resize_workspace_bytes.restype = sz
        L.moe_cache_resize_workspace_bytes.argtypes = [cp, i32]
        L.moe_cache_resize.restype = C.c_int
        L.moe_cache_resize.argtypes = [sp, cp, i32, vp, sz, vp]
        L.moe_cache_step.restype = C.c_int
        L.moe_cache_step.argtypes = [sp, cp, i32, vp, i32, pp, i32, vp]
        L.moe_ffn_workspace_bytes.restype = sz
        L.moe_ffn_workspace_bytes.argtypes = [sp, i32]
        L.moe_expert_ffn.restype = C.c_int
        L.moe_expert_ffn.argtypes = [sp, cp, i32, pp, vp, i32, vp, vp, vp, vp, sz, vp, vp]
        L.moe_layer_workspace_bytes.restype = sz
        L.moe_layer_workspace_bytes.argtypes = [sp, i32]
        L.moe_layer_forward.restype = C.c_int
        L.moe_layer_forward.argtypes = [sp, cp, i32, vp, i32, vp, vp, vp, pp, vp, vp, vp, sz,
                                        vp, vp]
        L.moe_prefill_workspace_bytes.restype = sz
        L.moe_prefill_workspace_bytes.argtypes = [sp, i32]
        L.moe_layer_prefetch.restype = C.c_int
        L.moe_layer_prefetch.argtypes = [sp, vp, i32, vp, vp]
        L.moe_expert_ffn_prefill.restype = C.c_int
        L.moe_expert_ffn_prefill.argtypes = [sp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp, vp]
        L.moe_layer_forward_prefill.restype = C.c_int
        L.moe_layer_forward_prefill.argtypes = [sp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz,
                                                vp, vp]
        L.moe_expert_ffn_noalloc.restype = C.c_int
        L.moe_expert_ffn_noalloc.argtypes = [sp, cp, i32, pp, vp, i32, vp, vp, vp, vp, vp]
        L.moe_profile_workspace_bytes.restype = sz
        L.moe_profile_workspace_bytes.argtypes = [sp]
        L.moe_profile_bandwidths.restype = C.c_int
        L.moe_profile_bandwidths.argtypes = [sp, cp, i32, vp, sz, i32, C.POINTER(i32),
                                             C.POINTER(i32), vp]
        _lib = L
    return _lib


# --------------------------------------------------------------- marshalling
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int) -> int:
    if rc != MOE_OK:
        raise MoeError(rc, moe_last_error())
    return rc


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


def moe_version() -> str:
    return lib().moe_version().decode()


def moe_expert_bytes(spec: MoeSpec) -> int:
    return int(lib().moe_expert_bytes(C.byref(spec)))


def moe_route(spec, x, T, w_router, bias, logits, ids, weights, stream=None):
    return _check(lib().moe_route(C.byref(spec), _ptr(x), T, _ptr(w_router), _ptr(bias),
                                  _ptr(logits), _ptr(ids), _ptr(weights), _stream(stream)))


def moe_cache_reset(spec, cache, stream=None):
    return _check(lib().moe_cache_reset(C.byref(spec), C.byref(cache), _stream(stream)))


def moe_debug_inject_ffn_stall(on=True):
    """Test hook: the next decode FFN call's gate/up kernel issues no copies, so its
    bounded waits run out and plan.err gets MOE_DERR_WAIT (include/moe.h)."""
    return _check(lib().moe_debug_inject_ffn_stall(1 if on else 0))


def moe_layer_kernel_count(spec, cache, T) -> int:
    return int(lib().moe_layer_kernel_count(C.byref(spec), C.byref(cache), T))


def moe_cache_place(spec, cache, ids, stream=None):
    """Preload the bank ids `ids` (host sequence of l*E + e) into the cache."""
    import numpy as np

    a = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).reshape(-1))
    return _check(lib().moe_cache_place(C.byref(spec), C.byref(cache),
                                        a.ctypes.data if a.size else None, int(a.size),
                                        _stream(stream)))


def moe_slots_for_budget(spec, free_bytes) -> int:
    n = int(lib().moe_slots_for_budget(C.byref(spec), int(free_bytes)))
    if n < 0:
        raise MoeError(MOE_EINVAL, moe_last_error())
    return n


def moe_cache_resize_workspace_bytes(cache, new_slots) -> int:
    return int(lib().moe_cache_resize_workspace_bytes(C.byref(cache), new_slots))


def moe_cache_resize(spec, cache, new_slots, workspace, workspace_bytes, stream=None):
    """Re-divide the slot pool into new_slots slots (cache.num_slots follows)."""
    return _check(lib().moe_cache_resize(C.byref(spec), C.byref(cache), new_slots,
                                         _ptr(workspace), workspace_bytes, _stream(stream)))


def moe_cache_step(spec, cache, layer, ids, T, plan, do_fill=1, stream=None):
    return _check(lib().moe_cache_step(C.byref(spec), C.byref(cache), layer, _ptr(ids), T,
                                       C.byref(plan), do_fill, _stream(stream)))


def moe_ffn_workspace_bytes(spec, T) -> int:
    return int(lib().moe_ffn_workspace_bytes(C.byref(spec), T))


def moe_expert_ffn(spec, cache, layer, plan, x, T, ids, weights, shared, workspace,
                   workspace_bytes, y, stream=None):
    return _check(lib().moe_expert_ffn(C.byref(spec), C.byref(cache), layer, C.byref(plan),
                                       _ptr(x), T, _ptr(ids), _ptr(weights), _ptr(shared),
                                       _ptr(workspace), workspace_bytes, _ptr(y),
                                       _stream(stream)))


def moe_expert_ffn_noalloc(spec, cache, layer, plan, x, T, ids, weights, shared, y, stream=None):
    """moe_expert_ffn without a workspace, for callers that cannot allocate device
    memory: the scratch is the library's built-in device array (see moe.h)."""
    return _check(lib().moe_expert_ffn_noalloc(C.byref(spec), C.byref(cache), layer,
                                               C.byref(plan), _ptr(x), T, _ptr(ids),
                                               _ptr(weights), _ptr(shared), _ptr(y),
                                               _stream(stream)))


def moe_layer_workspace_bytes(spec, T) -> int:
    return int(lib().moe_layer_workspace_bytes(C.byref(spec), T))


def moe_layer_forward(spec, cache, layer, x, T, w_router, bias, shared, plan, ids, weights,
                      workspace, workspace_bytes, y, stream=None):
    return _check(lib().moe_layer_forward(C.byref(spec), C.byref(cache), layer, _ptr(x), T,
                                          _ptr(w_router), _ptr(bias), _ptr(shared), C.byref(plan),
                                          _ptr(ids), _ptr(weights), _ptr(workspace),
                                          workspace_bytes, _ptr(y), _stream(stream)))


def moe_prefill_workspace_bytes(spec, T) -> int:
    return int(lib().moe_prefill_workspace_bytes(C.byref(spec), T))


def moe_profile_workspace_bytes(spec) -> int:
    return int(lib().moe_profile_workspace_bytes(C.byref(spec)))


def moe_profile_bandwidths(spec, cache, layer, workspace, workspace_bytes, reps=10, stream=None):
    """(B_P, B_H) in MB/s measured on the device (synchronises the stream)."""
    bp, bh = C.c_int32(0), C.c_int32(0)
    _check(lib().moe_profile_bandwidths(C.byref(spec), C.byref(cache), layer, _ptr(workspace),
                                        workspace_bytes, reps, C.byref(bp), C.byref(bh),
                                        _stream(stream)))
    return bp.value, bh.value


def moe_layer_prefetch(spec, bank, layer, dst, stream=None):
    return _check(lib().moe_layer_prefetch(C.byref(spec), _ptr(bank), layer, _ptr(dst),
                                           _stream(stream)))


def moe_expert_ffn_prefill(spec, layer_experts, x, T, ids, weights, shared, err, workspace,
                           workspace_bytes, y, stream=None):
    return _check(lib().moe_expert_ffn_prefill(C.byref(spec), _ptr(layer_experts), _ptr(x), T,
                                               _ptr(ids), _ptr(weights), _ptr(shared), _ptr(err),
                                               _ptr(workspace), workspace_bytes, _ptr(y),
                                               _stream(stream)))


def moe_layer_forward_prefill(spec, layer_experts, x, T, w_router, bias, shared, ids, weights,
                              err, workspace, workspace_bytes, y, stream=None):
    return _check(lib().moe_layer_forward_prefill(C.byref(spec), _ptr(layer_experts), _ptr(x), T,
                                                  _ptr(w_router), _ptr(bias), _ptr(shared),
                                                  _ptr(ids), _ptr(weights), _ptr(err),
                                                  _ptr(workspace), workspace_bytes, _ptr(y),
                                                  _stream(stream)))


# ------------------------------------------------- device memory (plumbing)
def make_spec(num_layers, hidden, inter, num_experts, top_k, router="softmax", n_groups=1,
              topk_groups=1, routed_scale=1.0, has_shared=False, shared_inter=None,
              fmt=FORMAT_INT4) -> MoeSpec:
    return MoeSpec(num_layers, hidden, inter, num_experts, top_k,
                   MOE_ROUTER_SIGMOID_GROUP if router == "sigmoid_group" else
                   MOE_ROUTER_SOFTMAX_TOPK, n_groups, topk_groups, routed_scale, 64,
                   1 if has_shared else 0, shared_inter if shared_inter else inter, fmt)


class DeviceCache:
    """Slot tables and slot pool in device memory (torch tensors) + the C struct."""

    def __init__(self, spec: MoeSpec, num_slots, k_victims, bp_mbps, bh_mbps, bank, device="cuda",
                 with_pool=True, policy=POLICY_SHARED_LRU, sync=True, capacity=None):
        import torch

        # capacity: slots the tables and the pool are allocated for (room for
        # moe_cache_resize to grow into); num_slots of them are in use
        cap = max(num_slots, capacity or 0)
        n_ids = spec.num_layers * spec.num_experts
        se = moe_expert_bytes(spec)
        self.slot_of_id = torch.full((n_ids,), -1, dtype=torch.int32, device=device)
        self.id_of_slot = torch.full((cap,), -1, dtype=torch.int32, device=device)
        self.ts = torch.zeros(cap, dtype=torch.int32, device=device)
        self.clock = torch.zeros(1, dtype=torch.int32, device=device)
        self.pool = (torch.empty((cap, se), dtype=torch.uint8, device=device)
                     if with_pool else None)
        self.bank = bank
        # sync words of the one-kernel decode layer step (None: the multi-kernel form)
        self.sync = (torch.zeros(CACHE_SYNC_WORDS, dtype=torch.int32, device=device)
                     if sync else None)
        self.c = MoeCache(num_slots, k_victims, bp_mbps, bh_mbps, _ptr(self.slot_of_id),
                          _ptr(self.id_of_slot), _ptr(self.ts), _ptr(self.clock),
                          _ptr(self.pool), _ptr(bank), policy, _ptr(self.sync))

    def host_tables(self):
        """slot_of_id, id_of_slot, ts, clock (the slots in use only)."""
        import numpy as np

        S = self.c.num_slots
        return (self.slot_of_id.cpu().numpy().copy(), self.id_of_slot[:S].cpu().numpy().copy(),
                self.ts[:S].cpu().numpy().view(np.uint32).copy(),
                self.clock.cpu().numpy().view(np.uint32).copy())


class DevicePlan:
    """Fixed-shape step buffers in device memory + the C struct."""

    NAMES = ("uniq", "hit_ids", "hit_slots", "fill_ids", "fill_slots", "evicted_ids",
             "direct_ids")

    def __init__(self, capacity, k_victims, device="cuda"):
        import torch

        self.capacity = capacity
        self.buf = {n: torch.full((capacity,), -1, dtype=torch.int32, device=device)
                    for n in self.NAMES}
        self.victims = torch.full((max(k_victims, 1),), -1, dtype=torch.int32, device=device)
        self.counts = torch.zeros(8, dtype=torch.int32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        b = self.buf
        self.c = MoePlan(capacity, _ptr(b["uniq"]), _ptr(b["hit_ids"]), _ptr(b["hit_slots"]),
                         _ptr(b["fill_ids"]), _ptr(b["fill_slots"]), _ptr(b["evicted_ids"]),
                         _ptr(b["direct_ids"]), _ptr(self.victims), _ptr(self.counts),
                         _ptr(self.err))

    def read(self, K):
        """Host copy of the plan in the oracle's dict format (test helper)."""
        c = [int(v) for v in self.counts.cpu()]
        n_uniq, n_hit, n_miss, q, n_fill, n_direct, n_vict, now = c
        h = {n: t.cpu().numpy() for n, t in self.buf.items()}
        return {
            "uniq": h["uniq"][:n_uniq].copy(), "hit_ids": h["hit_ids"][:n_hit].copy(),
            "hit_slots": h["hit_slots"][:n_hit].copy(), "fill_ids": h["fill_ids"][:n_fill].copy(),
            "fill_slots": h["fill_slots"][:n_fill].copy(),
            "evicted_ids": h["evicted_ids"][:n_fill].copy(),
            "direct_ids": h["direct_ids"][:n_direct].copy(),
            "victims": self.victims.cpu().numpy()[:K].copy(), "counts": self.counts.cpu().numpy(),
            "n_uniq": n_uniq, "n_hit": n_hit, "n_miss": n_miss, "q": q, "n_fill": n_fill,
            "n_direct": n_direct, "n_victims": n_vict, "now": now,
            "err": int(self.err.cpu()[0]),
        }
