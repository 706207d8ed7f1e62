"""Device buffers of one synthetic job, filled in place on the GPU.

Allocates, per the FSDP2 per-parameter storage the kernels work on:
  grads[k][p]   rank k's bf16 gradient of parameter p (its own allocation);
  shards[r][p]  rank r's fp32 shard of p, inside a guard band of canaries;
  gathered      the rank-major bf16 buffer, sentinel in every padding slot;
  params[p]     parameter p's bf16 storage, inside a guard band.
Values come from the seeded generator (synth.h) through libtide_synth.so.
Tensors hold bf16 bit patterns as int16.
"""
from __future__ import annotations

import torch

from . import SENTINEL_BF16, Workload, amp, device_lib, dim0_inner, numel

GUARD_F32 = 64    # canary elements on each side of an fp32 output (256 bytes)
GUARD_BF16 = 128  # canary elements on each side of a bf16 output (256 bytes)
CANARY_F32 = 0x7FA5A5A5   # a NaN pattern no kernel writes
CANARY_BF16 = 0x7FA5


def _i16(v: int) -> int:
    return v - 0x10000 if v >= 0x8000 else v


def _i32(v: int) -> int:
    return v - 0x100000000 if v >= 0x80000000 else v


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what}: cudaError {rc}")


def fill_bf16(t: torch.Tensor, key: int, first: int, sigma: float, outlier_every=0,
              outlier_mult=1.0, stream=None):
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    _check(device_lib().synth_fill_bf16_device(t.data_ptr(), t.numel(), key, first, amp(sigma),
                                               outlier_every, outlier_mult, s), "synth fill")


def fill_f32(t: torch.Tensor, key: int, first: int, sigma: float, stream=None):
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    _check(device_lib().synth_fill_f32_device(t.data_ptr(), t.numel(), key, first, amp(sigma), s),
           "synth fill f32")


class DeviceJob:
    def __init__(self, wl: Workload, layout, device="cuda", guard=True, fill=True, align=8):
        self.wl = wl
        self.layout = layout
        self.align = align  # offset alignment the layout was created with
        self.device = torch.device(device)
        N, P = wl.num_ranks, wl.num_params
        self.N, self.P = N, P
        self.dims = [dim0_inner(s) for s in wl.shapes]
        self.chunk = [-(-d0 // N) for d0, _ in self.dims]
        self.shard_numel = [c * inner for c, (_, inner) in zip(self.chunk, self.dims)]
        gf = GUARD_F32 if guard else 0
        gb = GUARD_BF16 if guard else 0
        self.gf, self.gb = gf, gb
        dev = self.device
        self.grads = [[torch.empty(numel(s), dtype=torch.int16, device=dev) for s in wl.shapes]
                      for _ in range(N)]
        self.shard_bufs = [[torch.full((n + 2 * gf,), _i32(CANARY_F32), dtype=torch.int32, device=dev)
                            for n in self.shard_numel] for _ in range(N)]
        self.shards = [[b[gf: b.numel() - gf].view(torch.float32) for b in row]
                       for row in self.shard_bufs]
        self.S = layout.block_numel
        self.gathered = torch.full((N * self.S,), _i16(SENTINEL_BF16), dtype=torch.int16, device=dev)
        self.param_bufs = [torch.full((numel(s) + 2 * gb,), _i16(CANARY_BF16), dtype=torch.int16,
                                      device=dev) for s in wl.shapes]
        self.params = [b[gb: b.numel() - gb] for b in self.param_bufs]
        if fill:
            self.fill_inputs()

    def fill_inputs(self):
        wl = self.wl
        for k in range(self.N):
            for p in range(self.P):
                g = self.grads[k][p]
                if g.numel() == 0:
                    continue
                if wl.zero_grad(k, p):
                    g.zero_()
                else:
                    fill_bf16(g, wl.grad_key(k, p), 0, wl.sigma, wl.outlier_every, wl.outlier_mult)
        for p in range(self.P):
            d0, inner = self.dims[p]
            c = self.chunk[p]
            o = self.layout.param_offset(p)
            for r in range(self.N):
                v = max(0, min(c, d0 - r * c)) * inner
                if v:
                    dst = self.gathered[r * self.S + o: r * self.S + o + v]
                    fill_bf16(dst, wl.gather_key(p), r * c * inner, wl.sigma)

    def make_pack_inputs(self):
        """fp32 shards filled from the generator (inputs of the AG pack),
        separate from the reduce-scatter outputs."""
        self.pack_src = [[torch.empty(n, dtype=torch.float32, device=self.device)
                          for n in self.shard_numel] for _ in range(self.N)]
        for r in range(self.N):
            for p in range(self.P):
                t = self.pack_src[r][p]
                if t.numel():
                    fill_f32(t, self.wl.shard_key(r, p), 0, self.wl.sigma)
        self.packed = torch.full((self.N * self.S,), _i16(SENTINEL_BF16), dtype=torch.int16,
                                 device=self.device)

    def make_slots(self):
        """One N*S bf16 slot per rank (the vacated all-gather buffers), sentinel-filled."""
        self.slots = [torch.full((self.N * self.S,), _i16(SENTINEL_BF16), dtype=torch.int16,
                                 device=self.device) for _ in range(self.N)]

    def pack_src_ptrs(self, rank=None):
        if rank is None:
            return [self.pack_src[r][p] for r in range(self.N) for p in range(self.P)]
        return [self.pack_src[rank][p] for p in range(self.P)]

    # pointer lists in the ABI's order
    def grad_ptrs(self):
        return [self.grads[k][p] for k in range(self.N) for p in range(self.P)]

    def shard_ptrs(self):
        return [self.shards[r][p] for r in range(self.N) for p in range(self.P)]

    def param_ptrs(self):
        return list(self.params)

    def guards_intact(self) -> bool:
        ok = True
        gf, gb = self.gf, self.gb
        if gf:
            for row in self.shard_bufs:
                for b in row:
                    ok &= bool((b[:gf] == _i32(CANARY_F32)).all()) and bool((b[b.numel() - gf:] == _i32(CANARY_F32)).all())
        if gb:
            for b in self.param_bufs:
                ok &= bool((b[:gb] == _i16(CANARY_BF16)).all()) and bool((b[b.numel() - gb:] == _i16(CANARY_BF16)).all())
        return ok

    def reset_outputs(self):
        for row in self.shard_bufs:
            for b in row:
                b.fill_(_i32(CANARY_F32))
        for b in self.param_bufs:
            b.fill_(_i16(CANARY_BF16))

    def nbytes(self) -> int:
        t = sum(g.numel() * 2 for row in self.grads for g in row)
        t += sum(b.numel() * 4 for row in self.shard_bufs for b in row)
        t += self.gathered.numel() * 2 + sum(b.numel() * 2 for b in self.param_bufs)
        return t
