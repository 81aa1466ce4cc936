"""Thin ctypes binding of include/dspark_walk.h (argument marshalling only).

The functions below carry the C names and do nothing but convert Python
arguments (torch tensors, ints, streams) to the C call and turn a negative
status into an exception.  Every step of the walk runs in the CUDA library;
there is no fallback: if the library is missing, loading it raises.
"""
import ctypes
import os

import torch

from . import _build

OK = 0
EINVAL = -1
ENOMEM = -2
ECUDA = -3
ETIMEOUT = -4
EANCHOR = -5
EUNSUPPORTED = -6
ETEMP = -7
ELIMIT = -8
EINTERNAL = -9

TRACE_SM_CLOCK = 0
TRACE_GLOBAL_TIMER = 1

KERNEL_STREAM = 0
KERNEL_RESIDENT = 1
KERNEL_BATCHED = 2

SEED_FIXED = 0
SEED_PER_ROUND = 1

SAMPLER_GUMBEL = 0
SAMPLER_GROUP = 1

CELL_MARKOV = 0
CELL_GATED = 1
CELL_RNN = 2
CELL_GRU = 3

_lib = None


class WalkError(RuntimeError):
    """A C-ABI call returned a negative status."""

    def __init__(self, code, where):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (where, dspark_walk_strerror(code), code))


class dspark_walk_plan(ctypes.Structure):
    _fields_ = [
        ("V", ctypes.c_int64), ("r", ctypes.c_int), ("n_cta", ctypes.c_int),
        ("threads", ctypes.c_int), ("rows_per_cta", ctypes.c_int),
        ("rows_tmem", ctypes.c_int), ("rows_smem", ctypes.c_int), ("rows_rf", ctypes.c_int),
        ("rows_stream", ctypes.c_int), ("resident_bytes", ctypes.c_int64),
        ("streamed_bytes", ctypes.c_int64), ("max_B", ctypes.c_int),
        ("max_gamma", ctypes.c_int), ("kernel", ctypes.c_int), ("sm_count", ctypes.c_int),
        ("weight_bytes", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


EXPORTS = [
    "dspark_walk_create", "dspark_walk_run", "dspark_walk_run_host", "dspark_walk_status",
    "dspark_walk_get_plan", "dspark_walk_set_limits", "dspark_walk_strerror",
    "dspark_walk_destroy", "dspark_walk_run_noalloc", "dspark_walk_set_kernel",
    "dspark_walk_set_trace", "dspark_walk_set_seed_mode", "dspark_walk_round",
    "dspark_walk_gumbel_noise", "dspark_walk_set_sampler", "dspark_walk_set_cell",
    "dspark_walk_set_state_output", "dspark_walk_unit_rates", "dspark_walk_set_trace_clock",
]


def library_path():
    return _build.LIB


def load(build_if_missing=True):
    """Load libdspark_walk.so (building it first if asked and missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise OSError("CUDA library %s is missing; run __graft_entry__.build()" % path)
        _build.build()
    L = ctypes.CDLL(path)
    vp, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
    L.dspark_walk_create.argtypes = [vp, vp, i64, i32, i32, i32, ctypes.POINTER(vp)]
    L.dspark_walk_run.argtypes = [vp, vp, vp, vp, u64, vp, i32, i32, vp, vp]
    L.dspark_walk_run_host.argtypes = [vp, vp, vp, vp, u64, vp, i32, i32, vp, vp]
    L.dspark_walk_status.argtypes = [vp, vp]
    L.dspark_walk_get_plan.argtypes = [vp, ctypes.POINTER(dspark_walk_plan)]
    L.dspark_walk_set_limits.argtypes = [vp, i64, i32]
    L.dspark_walk_strerror.argtypes = [i32]
    L.dspark_walk_strerror.restype = ctypes.c_char_p
    L.dspark_walk_destroy.argtypes = [vp]
    L.dspark_walk_set_kernel.argtypes = [vp, i32]
    L.dspark_walk_set_trace.argtypes = [vp, vp, i64]
    L.dspark_walk_set_trace_clock.argtypes = [vp, i32]
    L.dspark_walk_run_noalloc.argtypes = [vp, vp, i64, i32, vp, vp, vp, u64, vp, i32, i32, vp, vp]
    L.dspark_walk_set_seed_mode.argtypes = [vp, i32]
    L.dspark_walk_set_sampler.argtypes = [vp, i32]
    L.dspark_walk_set_cell.argtypes = [vp, i32, vp, vp]
    L.dspark_walk_set_state_output.argtypes = [vp, vp]
    L.dspark_walk_round.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint64)]
    L.dspark_walk_gumbel_noise.argtypes = [vp, vp, i64, vp]
    L.dspark_walk_unit_rates.argtypes = [ctypes.POINTER(ctypes.c_double), i32, vp]
    for name in EXPORTS:
        if name != "dspark_walk_strerror":
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc, where):
    if rc != OK:
        raise WalkError(rc, where)
    return rc


def dspark_walk_strerror(code):
    return load().dspark_walk_strerror(int(code)).decode()


def dspark_walk_create(W1, W2, V, r, max_B, max_gamma):
    """Create a walk over device bf16 W1, W2 [V, r]; returns the handle (int)."""
    h = ctypes.c_void_p()
    _check(load().dspark_walk_create(_ptr(W1), _ptr(W2), int(V), int(r), int(max_B),
                                     int(max_gamma), ctypes.byref(h)), "dspark_walk_create")
    return h.value


def dspark_walk_run(h, base_logits, anchor, temperature, seed, out_tokens, B, gamma,
                    out_logits=None, stream=None):
    """Launch one round on `stream` (default: torch's current stream)."""
    return _check(load().dspark_walk_run(
        h, _ptr(base_logits), _ptr(anchor), _ptr(temperature), int(seed) & (2**64 - 1),
        _ptr(out_tokens), int(B), int(gamma), _ptr(out_logits), _stream(stream)),
        "dspark_walk_run")


def dspark_walk_run_host(h, base_logits, anchor, temperature, seed, out_tokens, B, gamma,
                         out_logits=None, stream=None):
    """One round from host (CPU, ideally pinned) tensors; returns the device status."""
    return load().dspark_walk_run_host(
        h, _ptr(base_logits), _ptr(anchor), _ptr(temperature), int(seed) & (2**64 - 1),
        _ptr(out_tokens), int(B), int(gamma), _ptr(out_logits), _stream(stream))


def dspark_walk_status(h, stream=None):
    """Wait for the stream; return (and clear) the device status word."""
    return load().dspark_walk_status(h, _stream(stream))


def dspark_walk_get_plan(h):
    p = dspark_walk_plan()
    _check(load().dspark_walk_get_plan(h, ctypes.byref(p)), "dspark_walk_get_plan")
    return p.as_dict()


def dspark_walk_set_limits(h, timeout_ns, skip_cta=-1):
    return _check(load().dspark_walk_set_limits(h, int(timeout_ns), int(skip_cta)),
                  "dspark_walk_set_limits")


def dspark_walk_set_kernel(h, kernel):
    return _check(load().dspark_walk_set_kernel(h, int(kernel)), "dspark_walk_set_kernel")


def dspark_walk_set_seed_mode(h, mode):
    return _check(load().dspark_walk_set_seed_mode(h, int(mode)), "dspark_walk_set_seed_mode")


def dspark_walk_set_sampler(h, sampler):
    return _check(load().dspark_walk_set_sampler(h, int(sampler)), "dspark_walk_set_sampler")


def dspark_walk_set_cell(h, cell, M=None, X=None):
    """The serial head: CELL_MARKOV; CELL_GATED / CELL_RNN with M a device bf16
    [256, 256] tensor; CELL_GRU with M [768, 256] and the token tables X
    [3, V, 256] (referenced by the handle: keep them alive)."""
    for t in (M, X):
        if t is not None:
            assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
    return _check(load().dspark_walk_set_cell(h, int(cell), _ptr(M), _ptr(X)),
                  "dspark_walk_set_cell")


def dspark_walk_set_state_output(h, out_state=None):
    """Later runs write each step's latent into out_state (device bf16 [B, gamma, 256])."""
    if out_state is not None:
        assert out_state.is_cuda and out_state.dtype == torch.bfloat16
        assert out_state.is_contiguous()
    return _check(load().dspark_walk_set_state_output(h, _ptr(out_state)),
                  "dspark_walk_set_state_output")


def dspark_walk_round(h, stream=None):
    r = ctypes.c_uint64(0)
    _check(load().dspark_walk_round(h, _stream(stream), ctypes.byref(r)), "dspark_walk_round")
    return r.value


def dspark_walk_gumbel_noise(bits, noise, stream=None):
    """noise[i] = the kernels' Gumbel noise of Philox word bits[i] (device tensors)."""
    assert bits.is_cuda and noise.is_cuda and bits.numel() == noise.numel()
    assert bits.dtype in (torch.int32, torch.uint32) and noise.dtype == torch.float32
    return _check(load().dspark_walk_gumbel_noise(_ptr(bits), _ptr(noise), bits.numel(),
                                                  _stream(stream)), "dspark_walk_gumbel_noise")


UNIT_RATE_NAMES = ("hmma_rf_cycles", "hmma_smem_cycles", "tc_tmem_a_cycles",
                   "resident_step_projection_cycles", "sm_mhz", "tmem_ld_cycles_per_kb",
                   "tmem_fed_step_projection_cycles", None, "cross_sm_hop_ns",
                   "l2_load_round_trip_cycles")


def dspark_walk_unit_rates(stream=None):
    """The on-chip tier rates and the cross-SM latencies of the current device
    (see the header), as a dict."""
    out = (ctypes.c_double * len(UNIT_RATE_NAMES))()     # out[7] = 0: constant operands
    _check(load().dspark_walk_unit_rates(out, len(UNIT_RATE_NAMES), _stream(stream)),
           "dspark_walk_unit_rates")
    return {k: v for k, v in zip(UNIT_RATE_NAMES, list(out)) if k is not None}


def dspark_walk_set_trace(h, device_buffer, nbytes):
    return _check(load().dspark_walk_set_trace(h, _ptr(device_buffer), int(nbytes)),
                  "dspark_walk_set_trace")


def dspark_walk_set_trace_clock(h, clock):
    return _check(load().dspark_walk_set_trace_clock(h, int(clock)), "dspark_walk_set_trace_clock")


def dspark_walk_destroy(h):
    return _check(load().dspark_walk_destroy(h), "dspark_walk_destroy")


def dspark_walk_run_noalloc(W1, W2, V, r, base_logits, anchor, temperature, seed, out_tokens,
                            B, gamma, out_logits=None, stream=None):
    """One round without any device allocation (B <= 64, gamma <= 16).

    For callers that may not allocate device memory; W2 is read in place and
    the rendezvous slots are a fixed block inside the library.  Returns the
    launch status; device-detected errors show up as -1 tokens.
    """
    return _check(load().dspark_walk_run_noalloc(
        _ptr(W1), _ptr(W2), int(V), int(r), _ptr(base_logits), _ptr(anchor), _ptr(temperature),
        int(seed) & (2**64 - 1), _ptr(out_tokens), int(B), int(gamma), _ptr(out_logits),
        _stream(stream)), "dspark_walk_run_noalloc")


class Walk:
    """Owns one handle; weights are device bf16 tensors [V, 256]."""

    def __init__(self, W1, W2, max_B, max_gamma):
        assert W1.is_cuda and W2.is_cuda and W1.dtype == torch.bfloat16 == W2.dtype
        self.W1 = W1.contiguous()        # referenced by the handle: keep alive
        V, r = W2.shape
        self.V, self.r = V, r
        self.max_B, self.max_gamma = max_B, max_gamma
        self.h = dspark_walk_create(self.W1, W2.contiguous(), V, r, max_B, max_gamma)

    def plan(self):
        return dspark_walk_get_plan(self.h)

    def set_kernel(self, kernel):
        dspark_walk_set_kernel(self.h, kernel)

    def set_seed_mode(self, mode):
        dspark_walk_set_seed_mode(self.h, mode)

    def set_sampler(self, sampler):
        dspark_walk_set_sampler(self.h, sampler)

    def set_cell(self, cell, M=None, X=None):
        self.M = None if M is None else M.contiguous()      # referenced: keep alive
        self.X = None if X is None else X.contiguous()
        dspark_walk_set_cell(self.h, cell, self.M, self.X)

    def set_state_output(self, out_state=None):
        dspark_walk_set_state_output(self.h, out_state)

    def round(self, stream=None):
        return dspark_walk_round(self.h, stream)

    def run(self, base, anchor, temperature, seed, out_tokens=None, out_logits=None,
            stream=None):
        B, gamma, V = base.shape
        if out_tokens is None:
            out_tokens = torch.empty(B, gamma, dtype=torch.int32, device=base.device)
        dspark_walk_run(self.h, base, anchor, temperature, seed, out_tokens, B, gamma,
                        out_logits, stream)
        return out_tokens

    def status(self, stream=None):
        return dspark_walk_status(self.h, stream)

    def close(self):
        if self.h:
            dspark_walk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
