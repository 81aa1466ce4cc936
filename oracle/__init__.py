"""CPU oracle of DSpark's serial draft walk (fp64 projection): the Markov head and the
gated and RNN recurrent heads.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package.  It shares no code with the
CUDA library and never imports it.  The arithmetic lives in ``oracle.c``; this
module only marshals numpy arrays through ctypes.

Source of the method: "Keeping the Draft Walk on Chip: One Launch for DSpark's
Markov Head", sections "The serial part of a parallel drafter" (recurrence and
the rounding of W2 @ u), "The idea: make the walk resident" (ties to the
smallest id, Philox-keyed Gumbel-max), "B200: the bf16 table fits on chip"
(fp32 accumulation, two bf16 roundings); vLLM pull request #64442, section
"Details" (plain fp32 Gumbel noise; tokens follow softmax(logits / T)).

Every array of bf16 values is passed as its raw bits (numpy ``uint16``).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")


class OracleError(RuntimeError):
    """The oracle rejected its input (bad size, anchor or temperature)."""


class Oracle:
    """The oracle library at ``path`` (the default build unless a test asks)."""

    def __init__(self, path=None):
        path = path or _build.build()
        L = ctypes.CDLL(path)
        L.orc_bf16_rne_many.restype = None
        L.orc_bf16_rne_many.argtypes = [_f64p, _u16p, ctypes.c_int64]
        L.orc_philox_many.restype = None
        L.orc_philox_many.argtypes = [_u32p, _u32p, _u32p, ctypes.c_int64]
        L.orc_noise_bits.restype = ctypes.c_uint32
        L.orc_noise_bits.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
        L.orc_uniform.restype = ctypes.c_float
        L.orc_uniform.argtypes = [ctypes.c_uint32]
        L.orc_gumbel.restype = ctypes.c_float
        L.orc_gumbel.argtypes = [ctypes.c_float]
        L.orc_sample_score.restype = ctypes.c_float
        L.orc_sample_score.argtypes = [ctypes.c_uint16, ctypes.c_float, ctypes.c_float]
        L.orc_walk.restype = ctypes.c_int
        L.orc_walk.argtypes = [
            _u16p, _u16p, ctypes.c_int64, ctypes.c_int,
            _u16p, _i32p, _f32p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, _i32p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ]
        L.orc_walk2.restype = ctypes.c_int
        L.orc_walk2.argtypes = [
            _u16p, _u16p, ctypes.c_int64, ctypes.c_int,
            _u16p, _i32p, _f32p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int, _i32p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ]
        L.orc_walk3.restype = ctypes.c_int
        L.orc_walk3.argtypes = [
            _u16p, _u16p, ctypes.c_int64, ctypes.c_int,
            _u16p, _i32p, _f32p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, _i32p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ]
        L.orc_cell_update.restype = None
        L.orc_cell_update.argtypes = [ctypes.c_int, _u16p, ctypes.c_int, ctypes.c_void_p, _u16p,
                                      _u16p, ctypes.c_void_p]
        L.orc_group_uniforms.restype = None
        L.orc_group_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int64, ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_float)]
        self.L = L
        self.path = path

    def bf16_rne(self, x):
        """Round float64 values to bf16 (ties to even); returns uint16 bits."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.L.orc_bf16_rne_many(x.reshape(-1), out.reshape(-1), x.size)
        return out

    def philox4x32_10(self, ctr, key):
        """Philox4x32-10 on rows of ctr [n,4] and key [n,2] (uint32)."""
        ctr = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(-1, 4)
        key = np.ascontiguousarray(key, dtype=np.uint32).reshape(-1, 2)
        out = np.empty_like(ctr)
        self.L.orc_philox_many(ctr, key, out, ctr.shape[0])
        return out

    def noise_bits(self, seed, b, k, v):
        """The 32 random bits of token v, request b, step k."""
        return int(self.L.orc_noise_bits(seed, b, k, v))

    def uniform(self, x):
        """Random bits -> the fp32 uniform the walk uses."""
        return float(self.L.orc_uniform(x))

    def gumbel(self, U):
        """fp32 Gumbel noise -log(-log U)."""
        return float(self.L.orc_gumbel(U))

    def sample_score(self, logit_bits, T, g):
        """fp32 selection score fp32(logit / T) + g."""
        return float(self.L.orc_sample_score(logit_bits, T, g))

    def walk(self, W1, W2, base, anchor, temperature, seed, forced=None,
             want_logits=True, want_scores=False, nthreads=1, req0=0, sampler=0,
             want_groups=False):
        """Run the walk for every request.

        W1, W2: uint16 [V, r]; base: uint16 [B, gamma, V]; anchor: int32 [B];
        temperature: float32 [B]; forced: optional int32 [B, gamma] (step
        k > 0 takes prev = forced[b, k-1]); req0: request index of row 0 (row
        i draws request req0 + i's noise); sampler: 0 per-token Gumbel-max, 1
        group inverse-CDF.  Returns (tokens int32 [B, gamma], logits uint16
        [B, gamma, V] or None, scores float32 [B, gamma, V] or None), and with
        want_groups a 4th item (group scores float32, in-group picks int32,
        pick margins float32, each [B, gamma, ceil(V / 8)]).
        """
        W1 = np.ascontiguousarray(W1, dtype=np.uint16)
        W2 = np.ascontiguousarray(W2, dtype=np.uint16)
        base = np.ascontiguousarray(base, dtype=np.uint16)
        anchor = np.ascontiguousarray(anchor, dtype=np.int32)
        temperature = np.ascontiguousarray(temperature, dtype=np.float32)
        V, r = W2.shape
        if W1.shape != (V, r):
            raise ValueError("W1 and W2 must both be [V, r]")
        B, gamma, Vb = base.shape
        if Vb != V or anchor.shape != (B,) or temperature.shape != (B,):
            raise ValueError("base must be [B, gamma, V]; anchor and temperature [B]")
        tokens = np.zeros((B, gamma), dtype=np.int32)
        logits = np.zeros((B, gamma, V), dtype=np.uint16) if want_logits else None
        scores = np.zeros((B, gamma, V), dtype=np.float32) if want_scores else None
        ng = (V + 7) // 8
        groups = None
        if want_groups:
            groups = (np.zeros((B, gamma, ng), dtype=np.float32),
                      np.zeros((B, gamma, ng), dtype=np.int32),
                      np.zeros((B, gamma, ng), dtype=np.float32))
        forced_arr = None
        if forced is not None:
            forced_arr = np.ascontiguousarray(forced, dtype=np.int32)
            if forced_arr.shape != (B, gamma):
                raise ValueError("forced must be [B, gamma]")
        rc = self.L.orc_walk2(
            W1, W2, V, r, base, anchor, temperature, int(seed) & (2**64 - 1), B, gamma,
            int(req0), forced_arr.ctypes.data if forced_arr is not None else None,
            int(sampler), tokens,
            logits.ctypes.data if logits is not None else None,
            scores.ctypes.data if scores is not None else None,
            groups[0].ctypes.data if groups is not None else None,
            groups[1].ctypes.data if groups is not None else None,
            groups[2].ctypes.data if groups is not None else None,
            int(nthreads))
        if rc != 0:
            raise OracleError("oracle walk rejected its input (code %d)" % rc)
        if want_groups:
            return tokens, logits, scores, groups
        return tokens, logits, scores

    def walk_cell(self, W1, W2, base, anchor, temperature, seed, cell, M=None, forced=None,
                  forced_state=None, want_logits=True, want_scores=False, nthreads=1, req0=0,
                  sampler=0, want_groups=False, X=None):
        """A recurrent head's walk (cell 1 gated, 2 RNN, 3 GRU; 0 is the Markov head).

        M: uint16 [r, r] recurrent matrix ([3r, r] for the GRU); X: the GRU's
        token tables, uint16 [3, V, r]; forced_state: optional uint16
        [B, gamma, r] (step k updates from forced_state[b, k-1] and projects
        forced_state[b, k]).  Returns (tokens, logits, scores, states uint16
        [B, gamma, r], states_exact float64 [B, gamma, r]), and with want_groups a
        6th item as ``walk``'s 4th (sampler 1's group scores, picks, margins).
        """
        W1 = np.ascontiguousarray(W1, dtype=np.uint16)
        W2 = np.ascontiguousarray(W2, dtype=np.uint16)
        base = np.ascontiguousarray(base, dtype=np.uint16)
        anchor = np.ascontiguousarray(anchor, dtype=np.int32)
        temperature = np.ascontiguousarray(temperature, dtype=np.float32)
        V, r = W2.shape
        if W1.shape != (V, r):
            raise ValueError("W1 and W2 must both be [V, r]")
        B, gamma, Vb = base.shape
        if Vb != V or anchor.shape != (B,) or temperature.shape != (B,):
            raise ValueError("base must be [B, gamma, V]; anchor and temperature [B]")
        Mc = Xc = None
        if M is not None:
            Mc = np.ascontiguousarray(M, dtype=np.uint16)
            if Mc.shape != ((3 * r, r) if cell == 3 else (r, r)):
                raise ValueError("M must be [r, r] ([3r, r] for the GRU)")
        if X is not None:
            Xc = np.ascontiguousarray(X, dtype=np.uint16)
            if Xc.shape != (3, V, r):
                raise ValueError("X must be [3, V, r]")
        fs = None
        if forced_state is not None:
            fs = np.ascontiguousarray(forced_state, dtype=np.uint16)
            if fs.shape != (B, gamma, r):
                raise ValueError("forced_state must be [B, gamma, r]")
        forced_arr = None
        if forced is not None:
            forced_arr = np.ascontiguousarray(forced, dtype=np.int32)
            if forced_arr.shape != (B, gamma):
                raise ValueError("forced must be [B, gamma]")
        tokens = np.zeros((B, gamma), dtype=np.int32)
        logits = np.zeros((B, gamma, V), dtype=np.uint16) if want_logits else None
        scores = np.zeros((B, gamma, V), dtype=np.float32) if want_scores else None
        states = np.zeros((B, gamma, r), dtype=np.uint16)
        exact = np.zeros((B, gamma, r), dtype=np.float64)
        ng = (V + 7) // 8
        groups = None
        if want_groups:
            groups = (np.zeros((B, gamma, ng), dtype=np.float32),
                      np.zeros((B, gamma, ng), dtype=np.int32),
                      np.zeros((B, gamma, ng), dtype=np.float32))
        ptr = lambda a: a.ctypes.data if a is not None else None
        rc = self.L.orc_walk3(
            W1, W2, V, r, base, anchor, temperature, int(seed) & (2**64 - 1), B, gamma,
            int(req0), ptr(forced_arr), int(sampler), int(cell), ptr(Mc), ptr(Xc), ptr(fs), tokens,
            ptr(logits), ptr(scores),
            ptr(groups[0]) if groups else None, ptr(groups[1]) if groups else None,
            ptr(groups[2]) if groups else None, ptr(states), ptr(exact), int(nthreads))
        if rc != 0:
            raise OracleError("oracle walk rejected its input (code %d)" % rc)
        if want_groups:
            return tokens, logits, scores, states, exact, groups
        return tokens, logits, scores, states, exact

    def cell_update(self, cell, M, hprev, x):
        """One state update: (h bf16 bits [r], the fp64 values before rounding);
        for the GRU x holds the token's three table rows ([3r])."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        r = x.shape[0] // 3 if cell == 3 else x.shape[0]
        M = np.ascontiguousarray(M, dtype=np.uint16)
        hp = None if hprev is None else np.ascontiguousarray(hprev, dtype=np.uint16)
        h = np.zeros(r, np.uint16)
        ex = np.zeros(r, np.float64)
        self.L.orc_cell_update(int(cell), M, r, hp.ctypes.data if hp is not None else None, x, h,
                               ex.ctypes.data)
        return h, ex

    def group_uniforms(self, seed, b, k, j):
        """The two uniforms (U1, U2) of group j of request b at step k (sampler 1)."""
        u1, u2 = ctypes.c_float(), ctypes.c_float()
        self.L.orc_group_uniforms(int(seed) & (2**64 - 1), int(b), int(k), int(j),
                                  ctypes.byref(u1), ctypes.byref(u2))
        return u1.value, u2.value


_default = None


def default() -> Oracle:
    """The oracle built from ``oracle.c`` in this directory."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def bf16_to_f64(h):
    """bf16 bits -> float64 values (exact)."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne(x):
    return default().bf16_rne(x)


def philox4x32_10(ctr, key):
    return default().philox4x32_10(ctr, key)


def noise_bits(seed, b, k, v):
    return default().noise_bits(seed, b, k, v)


def uniform(x):
    return default().uniform(x)


def gumbel(U):
    return default().gumbel(U)


def sample_score(logit_bits, T, g):
    return default().sample_score(logit_bits, T, g)


def walk(*args, **kwargs):
    return default().walk(*args, **kwargs)


def walk_cell(*args, **kwargs):
    return default().walk_cell(*args, **kwargs)


CELL_MARKOV, CELL_GATED, CELL_RNN, CELL_GRU = 0, 1, 2, 3


def cpu_threads(nthreads):
    """How many threads ``walk(..., nthreads)`` will really use."""
    if nthreads > 0:
        return nthreads
    return os.cpu_count() or 1
