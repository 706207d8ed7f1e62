"""Seeded synthetic inputs shared by the oracle-side tests, the GPU parity
tests and the benchmark.

One definition of every input (synth.h) is compiled for the host
(libsynth_host.so) and for the device (libtide_synth.so).  This package
holds the workload shapes and the ctypes glue; it contains none of the
reduce-scatter or placement arithmetic.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
DEVICE_LIB = os.path.join(_HERE, "libtide_synth.so")

STREAM_GRAD = 1
STREAM_GATHER = 2
STREAM_ZERO = 3
STREAM_SWEEP = 4
STREAM_SHARD = 5

#: bf16 quiet-NaN payload written into every padding / alignment slot of a
#: gathered buffer; it must never reach a parameter.
SENTINEL_BF16 = 0x7FC1

_host = None
_dev = None


def host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            raise RuntimeError(f"{HOST_LIB} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(HOST_LIB)
        lib.synth_hash_host.restype = ctypes.c_uint64
        lib.synth_hash_host.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_key_host.restype = ctypes.c_uint64
        lib.synth_key_host.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                       ctypes.c_uint64]
        lib.synth_amp_host.restype = ctypes.c_float
        lib.synth_amp_host.argtypes = [ctypes.c_double]
        lib.synth_fill_bf16_host.restype = None
        lib.synth_fill_bf16_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                             ctypes.c_uint64, ctypes.c_float, ctypes.c_uint32,
                                             ctypes.c_float]
        lib.synth_gather_bf16_host.restype = None
        lib.synth_gather_bf16_host.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                               ctypes.c_uint64, ctypes.c_float, ctypes.c_uint32,
                                               ctypes.c_float]
        lib.synth_fill_f32_host.restype = None
        lib.synth_fill_f32_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                            ctypes.c_uint64, ctypes.c_float]
        _host = lib
    return _host


def device_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEVICE_LIB):
            raise RuntimeError(f"{DEVICE_LIB} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(DEVICE_LIB)
        lib.synth_fill_bf16_device.restype = ctypes.c_int
        lib.synth_fill_bf16_device.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_float, ctypes.c_uint32,
                                               ctypes.c_float, ctypes.c_void_p]
        lib.synth_set_u16_device.restype = ctypes.c_int
        lib.synth_set_u16_device.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint16,
                                             ctypes.c_void_p]
        lib.synth_fill_f32_device.restype = ctypes.c_int
        lib.synth_fill_f32_device.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                              ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p]
        _dev = lib
    return _dev


def hash64(key: int, ctr: int) -> int:
    return host_lib().synth_hash_host(key, ctr)


def key(seed: int, stream: int, a: int, b: int) -> int:
    return host_lib().synth_key_host(seed, stream, a, b)


def amp(sigma: float) -> float:
    return host_lib().synth_amp_host(sigma)


def numel(shape) -> int:
    n = 1
    for d in shape:
        n *= int(d)
    return n


def dim0_inner(shape):
    """(d0, inner) of a contiguous row-major tensor; a 0-dim scalar is [1]."""
    if len(shape) == 0:
        return 1, 1
    inner = 1
    for d in shape[1:]:
        inner *= int(d)
    return int(shape[0]), inner


@dataclass
class Workload:
    """Shapes and value recipe of one synthetic reduce-scatter / placement job."""

    name: str
    num_ranks: int
    shapes: list
    names: list
    sigma: float
    seed: int = 0
    outlier_every: int = 0
    outlier_mult: float = 1.0
    # expert groups: lists of parameter indices whose gradients are zero
    # together on a rank where that expert received no tokens
    zero_groups: list = field(default_factory=list)
    zero_pct: int = 0

    @property
    def num_params(self) -> int:
        return len(self.shapes)

    @property
    def scale(self) -> float:
        return 1.0 / self.num_ranks

    @property
    def psi(self) -> int:
        return sum(numel(s) for s in self.shapes)

    def rs_bytes(self) -> int:
        """Algorithmic bytes of one reduce-scatter: N bf16 reads + one fp32 write per element."""
        return 2 * self.num_ranks * self.psi + 4 * self.psi

    def ag_bytes(self) -> int:
        """Algorithmic bytes of one placement: one bf16 read + one bf16 write per element."""
        return 4 * self.psi

    def grad_key(self, rank: int, p: int) -> int:
        return key(self.seed, STREAM_GRAD, rank, p)

    def gather_key(self, p: int) -> int:
        return key(self.seed, STREAM_GATHER, p, 0)

    def zero_grad(self, rank: int, p: int) -> bool:
        """True when rank `rank` holds an all-zero gradient for parameter p."""
        if not self.zero_pct:
            return False
        for e, group in enumerate(self.zero_groups):
            if p in group:
                h = hash64(key(self.seed, STREAM_ZERO, rank, e), 0)
                return h % 100 < self.zero_pct
        return False

    # ---- host materialisation (small workloads only) ----
    def host_grad(self, rank: int, p: int) -> np.ndarray:
        n = numel(self.shapes[p])
        out = np.zeros(n, dtype=np.uint16)
        if n and not self.zero_grad(rank, p):
            host_lib().synth_fill_bf16_host(out.ctypes.data, n, self.grad_key(rank, p), 0,
                                            amp(self.sigma), self.outlier_every,
                                            self.outlier_mult)
        return out

    def host_grad_at(self, rank: int, p: int, idx: np.ndarray) -> np.ndarray:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.zeros(idx.size, dtype=np.uint16)
        if idx.size and not self.zero_grad(rank, p):
            host_lib().synth_gather_bf16_host(out.ctypes.data, idx.ctypes.data, idx.size,
                                              self.grad_key(rank, p), amp(self.sigma),
                                              self.outlier_every, self.outlier_mult)
        return out

    def host_param_value(self, p: int) -> np.ndarray:
        """Full bf16 value of parameter p behind the gathered buffer."""
        n = numel(self.shapes[p])
        out = np.zeros(n, dtype=np.uint16)
        if n:
            host_lib().synth_fill_bf16_host(out.ctypes.data, n, self.gather_key(p), 0,
                                            amp(self.sigma), 0, 1.0)
        return out

    def shard_key(self, rank: int, p: int) -> int:
        return key(self.seed, STREAM_SHARD, rank, p)

    def host_shard_f32(self, rank: int, p: int, n: int) -> np.ndarray:
        """fp32 values of rank `rank`'s shard of p (pack inputs), n elements."""
        out = np.zeros(n, dtype=np.float32)
        if n:
            host_lib().synth_fill_f32_host(out.ctypes.data, n, self.shard_key(rank, p), 0,
                                           amp(self.sigma))
        return out

    def host_param_value_at(self, p: int, idx: np.ndarray) -> np.ndarray:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.zeros(idx.size, dtype=np.uint16)
        if idx.size:
            host_lib().synth_gather_bf16_host(out.ctypes.data, idx.ctypes.data, idx.size,
                                              self.gather_key(p), amp(self.sigma), 0, 1.0)
        return out


def _llama_layer(name, n, hidden, kv, ffn, sigma, **kw):
    shapes = [(hidden, hidden), (kv, hidden), (kv, hidden), (hidden, hidden),
              (ffn, hidden), (ffn, hidden), (hidden, ffn), (hidden,), (hidden,)]
    names = ["q", "k", "v", "o", "gate", "up", "down", "attn_norm", "ffn_norm"]
    return Workload(name, n, shapes, names, sigma, **kw)


def tiny() -> Workload:
    """Tiny block: N=4; q,k,v,o [256,256]; w1,w3 [704,256]; w2 [256,704]; norm [250]."""
    shapes = [(256, 256)] * 4 + [(704, 256), (704, 256), (256, 704), (250,)]
    names = ["q", "k", "v", "o", "w1", "w3", "w2", "norm"]
    return Workload("tiny", 4, shapes, names, 0.01, seed=0)


def llama8b() -> Workload:
    """Llama-3.1-8B-shaped decoder layer, N=8."""
    return _llama_layer("llama8b_layer", 8, 4096, 1024, 14336, 1e-3)


def llama70b() -> Workload:
    """Llama-3.1-70B-shaped decoder layer, N=8, 1% outliers scaled by 100."""
    return _llama_layer("llama70b_layer", 8, 8192, 1024, 28672, 1e-3,
                        outlier_every=100, outlier_mult=100.0)


def llama70b_attn() -> Workload:
    """The attention projections of the 70B-shaped layer alone (q,o [8192,8192],
    k,v [1024,8192], N=8, same outliers): a 3.6 GB case of the same kernel
    shape for profiler captures."""
    w = llama70b()
    return Workload("llama70b_attn", 8, w.shapes[:4], w.names[:4], w.sigma,
                    outlier_every=w.outlier_every, outlier_mult=w.outlier_mult)


def moe() -> Workload:
    """Qwen3-30B-A3B-shaped MoE layer, N=16, 128 experts, ~30% unrouted per rank."""
    shapes = [(4096, 2048), (512, 2048), (512, 2048), (2048, 4096), (128, 2048)]
    names = ["q", "k", "v", "o", "router"]
    groups = []
    for e in range(128):
        base = len(shapes)
        shapes += [(768, 2048), (768, 2048), (2048, 768)]
        names += [f"e{e}.gate", f"e{e}.up", f"e{e}.down"]
        groups.append([base, base + 1, base + 2])
    shapes += [(2048,), (2048,)]
    names += ["attn_norm", "ffn_norm"]
    return Workload("qwen3_30b_a3b_moe_layer", 16, shapes, names, 1e-3,
                    zero_groups=groups, zero_pct=30)


def sweep(num_ranks: int, seed: int = 0, inner: int = 4096, rows_per_rank: int = 2048) -> Workload:
    """Rank sweep: [d0, inner] params, d0 uniform in 512..16384 and not a
    multiple of N, until every rank's fp32 shard holds rows_per_rank * inner
    elements; the last parameter has d0 = remaining_rows * N - 1."""
    kk = key(seed, STREAM_SWEEP, num_ranks, 0)
    shapes, used, i = [], 0, 0
    while True:
        d0 = 512 + hash64(kk, i) % (16384 - 512 + 1)
        i += 1
        if d0 % num_ranks == 0:
            continue
        c = -(-d0 // num_ranks)
        if used + c >= rows_per_rank:
            break
        shapes.append((d0, inner))
        used += c
    shapes.append(((rows_per_rank - used) * num_ranks - 1, inner))
    names = [f"w{i}" for i in range(len(shapes))]
    return Workload(f"rank_sweep_n{num_ranks}", num_ranks, shapes, names, 1e-3, seed=seed)


WORKLOADS = {
    "tiny": tiny,
    "llama8b": llama8b,
    "llama70b": llama70b,
    "moe": moe,
    "llama70b_attn": llama70b_attn,
    "sweep16": lambda: sweep(16),
    "sweep32": lambda: sweep(32),
    "sweep64": lambda: sweep(64),
    # the N = 64 sweep's recipe with [d0, 1024] parameters and 448 rows per
    # rank: 3.8 GB of gradients, a profiler-sized case of the same kernels
    "sweep64_small": lambda: sweep(64, inner=1024, rows_per_rank=448),
}


def custom(name, num_ranks, shapes, sigma=0.01, seed=0) -> Workload:
    return Workload(name, num_ranks, list(shapes), [f"p{i}" for i in range(len(shapes))],
                    sigma, seed=seed)
