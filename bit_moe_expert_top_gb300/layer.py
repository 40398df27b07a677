"""One routed-expert FFN layer driven through libmoe's C ABI.

``MoELayer`` owns the device copies of a layer's expert weights (torch
allocations) and chains the library calls of one step:

    moe_route -> moe_permute -> FC1+SwiGLU -> FC2 -> moe_combine

with the weight path chosen by the layer's format:

* ``w2``    2-bit codebook experts (``moe_w2_mm``);
* ``mixed`` 2-bit base plus an FP4 delta cache: experts with a cache slot go
            through ``moe_mxfp4_mm``, the others through ``moe_w2_mm``
            (optionally split by group size: one row on the table GEMV, more
            on the tensor core);
* ``fp8``   MXFP4 experts converted per expert batch into a reused FP8
            workspace ring (``mxfp4_to_fp8_ws`` on a side stream) ahead of the
            FP8 matmuls on the main stream, the conversion of the next batch
            overlapping the matmuls of the current one ("国产GPU完成MoE大模型
            Day-0适配" §四);
* ``mxfp4`` the same MXFP4 experts multiplied as they are stored (E2M1
            codes and E8M0 scales straight into the block-scaled tensor core),
            no workspace;
* ``w2host`` 2-bit experts kept in pinned host memory with a device pool of
            resident slots plus staging slots: every step the routed experts
            that are not resident are copied over the CPU-GPU link into the
            staging slots (moe_stage_select + moe_cache_fill on a side
            stream) while the resident experts' FC1 runs (moe_w2_mm_slots).

The FP8 formats quantise the token rows to MXFP8 in the gather, and FC1
writes h as MXFP8 for FC2 ("FC1 + SwiGLU + MXFP8 quant, FC2").

No arithmetic happens here: every step runs in the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import _lib as L


def _dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


@dataclass
class StepBuffers:
    ids: torch.Tensor
    w: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    inv: torch.Tensor
    h: torch.Tensor
    h_scale: Optional[torch.Tensor]
    y: torch.Tensor
    out: torch.Tensor
    x_perm: Optional[torch.Tensor]
    x_perm_scale: Optional[torch.Tensor]
    dev_err: torch.Tensor
    ws: Optional[torch.Tensor] = None
    pws: Optional[torch.Tensor] = None   # grouping scratch of large steps (multi-CTA)
    fws: Optional[torch.Tensor] = None   # scratch of the fused FC1+FC2 launch
    h8: Optional[torch.Tensor] = None    # mixed with cache_fp8: the cache experts' h as MXFP8 codes
    h8_scale: Optional[torch.Tensor] = None


class MoELayer:
    def __init__(self, fmt: str, E: int, H: int, I: int, k: int, device="cuda", *,
                 w2=None, mx=None, expert_slot=None, fp8_batch: int = 64, fp8_ring: int = 2,
                 out_fmt: int = L.FMT_F32, mode: int = L.MODE_AUTO, gemm_min_rows: int = 2048,
                 resident=None, stage_slots: int = 64, fused: bool = True, split: bool = False,
                 side_sms: Optional[int] = None, single_launch: bool = True, cache_fp8: bool = False):
        """Weights are canonical host arrays (see synth.py / include/moe.h):
        w2 = (codes1, scales1, codes2, scales2) stacked over experts;
        mx = (q1, s1, q2, s2) stacked over cache slots (mixed) or experts (fp8);
        expert_slot int32 [E] (mixed): cache slot of each expert, -1 if none.
        fp8_batch / fp8_ring (fp8): experts per workspace batch and batches in
        the ring (default 64 x 2: 5.6 GB at H=7168, I=2048; per step 8.31 ms
        against 8.55 ms with 16 per batch, fewer persistent launch tails).
        resident (w2host): the expert ids kept in device memory; stage_slots:
        staging slots for the routed host-resident experts of one step.
        fused (w2, decode-sized steps on the table GEMV): FC1 and FC2 in one
        cooperative launch (moe_w2_decode_fused) instead of two calls; the
        default (measured ~1.5 % faster per decode step).
        split (mixed, tensor-core cache path): the 2-bit experts' calls in
        MOE_MODE_SPLIT (one-row groups on the table GEMV, larger ones on the
        tensor core); off by default: at 64 tokens (~2.8 rows per touched
        2-bit expert) it measured 6 % slower than the table GEMV alone.
        single_launch (w2 with fused, T*k <= 256, k <= 16, E <= 1024): the
        whole step (routing, grouping, FC1 + FC2, combine) as one launch of
        moe_w2_decode_layer instead of four calls; bit-identical outputs;
        the default (measured 5 % faster per decode step).
        cache_fp8 (mixed): the delta-cache (MXFP4) experts on the block-scaled
        FP8 tensor core with MXFP8 tokens and an MXFP8 h (their rows in the
        fp8 profile; the 2-bit experts stay in bf16); off by default, which
        keeps the whole layer in the bf16 profile.
        side_sms (fp8 on the tensor-core path, w2host): SMs reserved for the
        side-stream copy (the workspace conversion of the next batches, the
        staging of host-resident experts) while the matmuls run on the
        others (moe_set_side_sms); 0: copy and matmul each take the whole GPU
        in turn.  Default: 16 for w2host (the copy is bound by the CPU-GPU
        link, which 16 SMs keep full; measured 10 % faster per decode step),
        0 for fp8 (one SM converts only ~47 GB/s: every count measured
        slower)."""
        self.fmt, self.E, self.H, self.I, self.k = fmt, E, H, I, k
        self.device = torch.device(device)
        self.out_fmt, self.mode = out_fmt, mode
        self.fused = fused and fmt == "w2"
        self.single_launch = single_launch and self.fused
        self.split = split and fmt == "mixed"
        self.cache_fp8 = cache_fp8 and fmt == "mixed"
        self.side_sms = side_sms if side_sms is not None else (16 if fmt == "w2host" else 0)
        self.gemm_min_rows = gemm_min_rows
        dev = self.device
        if fmt in ("w2", "mixed", "w2host"):
            c1, s1, c2, s2 = w2
            self.c1k = torch.empty(c1.shape, dtype=torch.uint8, device=dev)
            self.s1k = torch.empty(s1.shape, dtype=torch.int16, device=dev)
            self.c2k = torch.empty(c2.shape, dtype=torch.uint8, device=dev)
            self.s2k = torch.empty(s2.shape, dtype=torch.int16, device=dev)
            for src_c, src_s, dc, ds, K in ((c1, s1, self.c1k, self.s1k, H), (c2, s2, self.c2k, self.s2k, I)):
                tc = _dev(src_c, dev)
                ts = _dev(src_s.view(np.int16), dev)
                L.moe_w2_repack(tc, ts, src_c.shape[0], src_c.shape[1], K, dc, ds)
                del tc, ts
        if fmt == "w2host":
            self._host_pool(resident, stage_slots)
        if fmt in ("mixed", "fp8", "mxfp4"):
            q1, s1, q2, s2 = mx
            self.q1, self.e1 = _dev(q1, dev), _dev(s1, dev)
            self.q2, self.e2 = _dev(q2, dev), _dev(s2, dev)
        self.expert_slot = None
        if fmt == "mixed":
            self.expert_slot = _dev(np.asarray(expert_slot, dtype=np.int32), dev)
        if fmt == "fp8":
            self.batch = fp8_batch
            self.ring = fp8_ring
            nslots = fp8_batch * fp8_ring
            self.ws1 = torch.empty((nslots, 2 * I, H), dtype=torch.uint8, device=dev)
            self.ws2 = torch.empty((nslots, H, I), dtype=torch.uint8, device=dev)
            e = np.arange(E)
            slot = ((e // fp8_batch) % fp8_ring) * fp8_batch + (e % fp8_batch)
            self.ws_slot = _dev(slot.astype(np.int32), dev)
            self.batch_experts = [_dev(np.arange(b, min(E, b + fp8_batch), dtype=np.int32), dev)
                                  for b in range(0, E, fp8_batch)]
            self.batch_slots = [self.ws_slot[b:min(E, b + fp8_batch)].contiguous() for b in range(0, E, fp8_batch)]
            self.conv_stream = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize(dev)

    def _host_pool(self, resident, stage_slots):
        """w2l weights of every expert to pinned host memory; the device keeps
        a pool of R resident slots + S staging slots."""
        E, dev = self.E, self.device
        full = [self.c1k, self.s1k, self.c2k, self.s2k]
        self.store = [t.cpu().pin_memory() for t in full]
        res = np.asarray(sorted(set(int(e) for e in (resident if resident is not None else []))), dtype=np.int64)
        self.R, self.S = int(res.size), int(stage_slots)
        self.pool = []
        for t in full:
            p = torch.empty((self.R + self.S,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev)
            if self.R:
                p[:self.R].copy_(t[torch.from_numpy(res).to(dev)])
            self.pool.append(p)
        self.c1k, self.s1k, self.c2k, self.s2k = self.pool
        self.pool_bytes = [t[0].numel() * t.element_size() for t in self.pool]
        rs = np.full(E, -1, dtype=np.int32)
        rs[res] = np.arange(self.R, dtype=np.int32)
        self.res_slot = _dev(rs, dev)
        self.weight_slot = torch.empty(E, dtype=torch.int32, device=dev)
        self.staged = torch.empty(self.S, dtype=torch.int32, device=dev)
        self.copy_stream = torch.cuda.Stream(device=dev)
        del full

    def staged_bytes(self, offsets: np.ndarray) -> int:
        """Bytes the step copies over the CPU-GPU link (w2host): the routed
        experts without a resident slot."""
        cnt = np.diff(np.asarray(offsets))
        rs = self.res_slot.cpu().numpy()
        n = int(np.sum((cnt > 0) & (rs < 0)))
        return min(n, self.S) * sum(self.pool_bytes)

    # ------------------------------------------------------------ buffers
    def use_gemm(self, T: int) -> bool:
        """Prefill-sized 2-bit and FP8-workspace steps run FC1/FC2 on the
        tensor cores over permuted (gathered) activation rows; decode-sized
        ones on the CUDA-core kernels.  Direct MXFP4 steps always use the
        block-scaled tensor core."""
        if self.fmt == "mxfp4":
            return True
        if self.fmt not in ("w2", "fp8") or self.mode == L.MODE_GEMV:
            return False
        return self.mode == L.MODE_GEMM or T * self.k >= self.gemm_min_rows

    def mx_tensor_path(self) -> bool:
        """Delta-cache (MXFP4) experts of a mixed layer run on the tensor-core
        kernel over gathered bf16 rows (any group size), unless GEMV mode is
        forced or the shape is not one it takes."""
        return (self.fmt == "mixed" and self.mode != L.MODE_GEMV and self.I % 128 == 0 and self.H % 256 == 0
                and self.H % 64 == 0 and self.I % 64 == 0)

    def buffers(self, T: int) -> StepBuffers:
        dev, E, H, I, k = self.device, self.E, self.H, self.I, self.k
        A = T * k
        gather = self.use_gemm(T)
        fp8 = self.fmt in ("fp8", "mxfp4")  # MXFP8 codes + scales for x_perm and h
        return StepBuffers(
            ids=torch.empty((T, k), dtype=torch.int32, device=dev),
            w=torch.empty((T, k), dtype=torch.float32, device=dev),
            offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            perm=torch.empty(A, dtype=torch.int32, device=dev),
            inv=torch.empty(A, dtype=torch.int32, device=dev),
            h=torch.empty((A, I), dtype=torch.uint8 if fp8 else torch.int16, device=dev),
            h_scale=torch.empty((A, I // 32), dtype=torch.uint8, device=dev) if fp8 else None,
            y=torch.empty((A, H), dtype=torch.int16, device=dev),
            out=torch.empty((T, H), dtype=torch.float32 if self.out_fmt == L.FMT_F32 else torch.int16, device=dev),
            x_perm=(torch.empty((A, H), dtype=torch.uint8, device=dev) if fp8 or self.cache_fp8 else
                    torch.empty((A, H), dtype=torch.int16, device=dev)
                    if gather or self.fmt == "fp8" or self.mx_tensor_path() else None),
            x_perm_scale=torch.empty((A, H // 32), dtype=torch.uint8, device=dev) if fp8 or self.cache_fp8 else None,
            dev_err=torch.zeros(1, dtype=torch.int32, device=dev),
            ws=self._gemv_ws(A) if self.fmt in ("w2", "mixed", "w2host") and not gather else None,
            pws=self._permute_ws(T),
            fws=self._fused_ws(A) if self.fused and not gather else None,
            h8=torch.empty((A, I), dtype=torch.uint8, device=dev) if self.cache_fp8 else None,
            h8_scale=torch.empty((A, I // 32), dtype=torch.uint8, device=dev) if self.cache_fp8 else None,
        )

    def _fused_ws(self, A: int) -> Optional[torch.Tensor]:
        """The fused launch's workspace: a barrier counter that starts at
        zero (the launch leaves it at zero), then the table GEMV's scratch."""
        n = L.moe_w2_decode_fused_workspace_size(A, self.H, self.I)
        return torch.zeros((n + 3) // 4, dtype=torch.int32, device=self.device) if n else None

    def _permute(self, b: StepBuffers, **kw):
        """moe_permute with the step's grouping scratch (multi-CTA when large)."""
        n = 0 if b.pws is None else b.pws.numel() * b.pws.element_size()
        L.moe_permute(b.ids, self.E, b.offsets, b.perm, b.inv, ws=b.pws, ws_bytes=n, **kw)

    def _permute_ws(self, T: int) -> Optional[torch.Tensor]:
        n = L.moe_permute_workspace_size(T, self.k, self.E)
        return torch.empty((n + 3) // 4, dtype=torch.int32, device=self.device) if n else None

    def _gemv_ws(self, A: int, cap_bytes: int = 1 << 30) -> Optional[torch.Tensor]:
        """Scratch of the 2-bit decode GEMV (FC1 and FC2 share it: the calls
        run one after the other on the stream; no initial contents needed).  Decode-sized steps
        need a few MB; beyond `cap_bytes` the GEMV runs without scratch."""
        n = max(L.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, A, self.I, self.H),
                L.moe_w2_mm_workspace_size(L.STAGE_FC2, A, self.H, self.I))
        if n > cap_bytes:
            return None
        return torch.empty((n + 3) // 4, dtype=torch.int32, device=self.device)

    # ------------------------------------------------------------ one step
    def step(self, x: torch.Tensor, logits: torch.Tensor, b: StepBuffers, ev: Optional[list] = None) -> torch.Tensor:
        """x: bf16 bit patterns int16 [T, H]; logits float32 [T, E].

        ``ev``: if given, a CUDA event pair is recorded around every expert
        matmul launch and appended as (label, start, end)."""
        T = x.shape[0]
        self._ev = ev
        E, H, I, k = self.E, self.H, self.I, self.k
        if self.single_launch and (T == 0 or b.fws is not None) and T * k <= 256 and k <= 16 and E <= 1024:
            with self._timed("w2_layer_single_launch"):
                L.moe_w2_decode_layer(logits, x, k, self.c1k, self.s1k, self.c2k, self.s2k, H, I, b.ids, b.w,
                                      b.offsets, b.perm, b.inv, b.h, b.y, b.out, self.out_fmt, b.fws,
                                      dev_err=b.dev_err)
            return b.out
        L.moe_route(logits, k, b.ids, b.w, b.dev_err)
        if self.fmt == "fp8":
            tc = self.use_gemm(T)
            self._permute(b, x=x, act_fmt=L.FMT_MXFP8, x_perm=b.x_perm,
                          x_perm_scale=b.x_perm_scale, dev_err=b.dev_err)
            self._fp8_experts(b, tc)
        elif self.fmt == "mxfp4":
            self._permute(b, x=x, act_fmt=L.FMT_MXFP8, x_perm=b.x_perm,
                          x_perm_scale=b.x_perm_scale, dev_err=b.dev_err)
            with self._timed("mx4_fc1_gemm"):
                L.moe_mxfp4_mm(L.STAGE_FC1_SWIGLU, b.x_perm, L.FMT_MXFP8, b.offsets, E, I, H, b.h, L.FMT_MXFP8,
                               e2m1=self.q1, e8m0=self.e1, act_scale=b.x_perm_scale, out_scale=b.h_scale,
                               mode=L.MODE_GEMM, dev_err=b.dev_err)
            with self._timed("mx4_fc2_gemm"):
                L.moe_mxfp4_mm(L.STAGE_FC2, b.h, L.FMT_MXFP8, b.offsets, E, H, I, b.y, L.FMT_BF16,
                               e2m1=self.q2, e8m0=self.e2, act_scale=b.h_scale, mode=L.MODE_GEMM,
                               dev_err=b.dev_err)
        elif self.fmt == "w2host":
            self._host_step(x, b)
        elif self.use_gemm(T):
            self._permute(b, x=x, act_fmt=L.FMT_BF16, x_perm=b.x_perm,
                          dev_err=b.dev_err)
            with self._timed("w2_fc1_gemm"):
                L.moe_w2_mm(L.STAGE_FC1_SWIGLU, b.x_perm, L.FMT_BF16, self.c1k, self.s1k, b.offsets, E, I, H, b.h,
                            L.FMT_BF16, mode=L.MODE_GEMM, dev_err=b.dev_err)
            with self._timed("w2_fc2_gemm"):
                L.moe_w2_mm(L.STAGE_FC2, b.h, L.FMT_BF16, self.c2k, self.s2k, b.offsets, E, H, I, b.y, L.FMT_BF16,
                            mode=L.MODE_GEMM, dev_err=b.dev_err)
        else:
            mx_tc = self.mx_tensor_path()
            if self.cache_fp8:  # the cache experts' matmuls read gathered MXFP8 rows
                self._permute(b, x=x, act_fmt=L.FMT_MXFP8, x_perm=b.x_perm, x_perm_scale=b.x_perm_scale,
                              dev_err=b.dev_err)
            elif mx_tc:  # the cache experts' matmuls read gathered rows
                self._permute(b, x=x, act_fmt=L.FMT_BF16, x_perm=b.x_perm,
                              dev_err=b.dev_err)
            else:
                self._permute(b, dev_err=b.dev_err)
            if b.fws is not None:  # FC1 and FC2 in one cooperative launch
                with self._timed("w2_fc1_fc2_fused"):
                    L.moe_w2_decode_fused(x, self.c1k, self.s1k, self.c2k, self.s2k, b.offsets, E, H, I, b.h, b.y,
                                          L.FMT_BF16, b.fws, act_row=b.perm, act_row_div=k, dev_err=b.dev_err)
                L.moe_combine(b.y, L.FMT_BF16, b.w, b.inv, T, k, H, b.out, self.out_fmt)
                return b.out
            # split: 2-bit experts of a mixed layer on gathered rows, single-row groups
            # on the table GEMV, larger ones on the tensor core (one pass over their weights)
            split = mx_tc and self.split and not self.cache_fp8
            w2_mode = (L.MODE_SPLIT if self.mode == L.MODE_AUTO else self.mode) if split else self.mode
            with self._timed("w2_fc1"):
                if split:
                    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, b.x_perm, L.FMT_BF16, self.c1k, self.s1k, b.offsets, E, I, H,
                                b.h, L.FMT_BF16, expert_slot=self.expert_slot, mode=w2_mode, ws=b.ws,
                                dev_err=b.dev_err)
                else:
                    L.moe_w2_mm(L.STAGE_FC1_SWIGLU, x, L.FMT_BF16, self.c1k, self.s1k, b.offsets, E, I, H, b.h,
                                L.FMT_BF16, act_row=b.perm, act_row_div=k, expert_slot=self.expert_slot,
                                mode=self.mode, ws=b.ws, dev_err=b.dev_err)
            if self.cache_fp8:
                with self._timed("mx_fc1"):
                    L.moe_mxfp4_mm(L.STAGE_FC1_SWIGLU, b.x_perm, L.FMT_MXFP8, b.offsets, E, I, H, b.h8, L.FMT_MXFP8,
                                   e2m1=self.q1, e8m0=self.e1, expert_slot=self.expert_slot,
                                   act_scale=b.x_perm_scale, out_scale=b.h8_scale, mode=L.MODE_GEMM,
                                   dev_err=b.dev_err)
            elif self.fmt == "mixed" and mx_tc:
                with self._timed("mx_fc1"):
                    L.moe_mxfp4_mm(L.STAGE_FC1_SWIGLU, b.x_perm, L.FMT_BF16, b.offsets, E, I, H, b.h, L.FMT_BF16,
                                   e2m1=self.q1, e8m0=self.e1, expert_slot=self.expert_slot, mode=L.MODE_GEMM,
                                   dev_err=b.dev_err)
            elif self.fmt == "mixed":
                with self._timed("mx_fc1"):
                    L.moe_mxfp4_mm(L.STAGE_FC1_SWIGLU, x, L.FMT_BF16, b.offsets, E, I, H, b.h, L.FMT_BF16,
                                   e2m1=self.q1, e8m0=self.e1, act_row=b.perm, act_row_div=k,
                                   expert_slot=self.expert_slot, mode=self.mode, dev_err=b.dev_err)
            with self._timed("w2_fc2"):
                L.moe_w2_mm(L.STAGE_FC2, b.h, L.FMT_BF16, self.c2k, self.s2k, b.offsets, E, H, I, b.y, L.FMT_BF16,
                            expert_slot=self.expert_slot, mode=w2_mode, ws=b.ws, dev_err=b.dev_err)
            if self.cache_fp8:
                with self._timed("mx_fc2"):
                    L.moe_mxfp4_mm(L.STAGE_FC2, b.h8, L.FMT_MXFP8, b.offsets, E, H, I, b.y, L.FMT_BF16,
                                   e2m1=self.q2, e8m0=self.e2, expert_slot=self.expert_slot,
                                   act_scale=b.h8_scale, mode=L.MODE_GEMM, dev_err=b.dev_err)
            elif self.fmt == "mixed":
                with self._timed("mx_fc2"):
                    L.moe_mxfp4_mm(L.STAGE_FC2, b.h, L.FMT_BF16, b.offsets, E, H, I, b.y, L.FMT_BF16,
                                   e2m1=self.q2, e8m0=self.e2, expert_slot=self.expert_slot,
                                   mode=L.MODE_GEMM if mx_tc else self.mode, dev_err=b.dev_err)
        L.moe_combine(b.y, L.FMT_BF16, b.w, b.inv, T, k, H, b.out, self.out_fmt)
        return b.out

    def _host_step(self, x, b: StepBuffers):
        """Grouping, staging of the routed host-resident experts on a side
        stream, FC1 over the resident experts meanwhile, FC1 over the staged
        ones once their copy has landed, then FC2 over all (table GEMV).
        With side SMs (``side_sms``) the copy holds a few SMs and the resident
        experts' FC1 and FC2 both run beside it on the others; the staged
        experts' FC1 and FC2 follow once it has landed."""
        E, H, I, k, R, S = self.E, self.H, self.I, self.k, self.R, self.S
        self._permute(b, dev_err=b.dev_err)
        L.moe_stage_select(b.offsets, self.res_slot, R, self.weight_slot, self.staged, dev_err=b.dev_err)
        main = torch.cuda.current_stream(self.device)
        cs = self.copy_stream
        cs.wait_stream(main)
        side = self.side_sms > 0
        prev = L.moe_set_side_sms(self.side_sms) if side else None
        try:
            L.moe_cache_fill(self.staged, self.store, [p[R:] for p in self.pool], self.pool_bytes, stream=cs)
            landed = torch.cuda.Event()
            landed.record(cs)

            def fc1(lo, hi):
                L.moe_w2_mm_slots(L.STAGE_FC1_SWIGLU, x, self.c1k, self.s1k, b.offsets, self.weight_slot, lo, hi, E,
                                  I, H, b.h, L.FMT_BF16, b.ws, act_row=b.perm, act_row_div=k, dev_err=b.dev_err)

            def fc2(lo, hi):
                L.moe_w2_mm_slots(L.STAGE_FC2, b.h, self.c2k, self.s2k, b.offsets, self.weight_slot, lo, hi, E, H, I,
                                  b.y, L.FMT_BF16, b.ws, dev_err=b.dev_err)

            if side:
                with self._timed("w2_resident"):
                    if R:
                        fc1(0, R)
                        fc2(0, R)
                with self._timed("w2_staged"):
                    main.wait_event(landed)
                    fc1(R, R + S)
                    fc2(R, R + S)
            else:
                with self._timed("w2_fc1"):
                    if R:
                        fc1(0, R)
                    main.wait_event(landed)
                    fc1(R, R + S)
                with self._timed("w2_fc2"):
                    fc2(0, R + S)
        finally:
            if prev is not None:
                L.moe_set_side_sms(prev)

    def capture(self, T: int) -> "LayerGraph":
        """The whole layer step for T tokens captured once into a CUDA graph
        (route, permute, the expert matmuls, combine: one graph launch per
        step, with the library's programmatic launch edges kept); see
        LayerGraph."""
        return LayerGraph(self, T)

    class _Timer:
        """Event pair around one library call; recorded as timing nodes when
        the step is being captured into a CUDA graph (external events)."""

        def __init__(self, ev, label):
            self.ev, self.label = ev, label

        @staticmethod
        def _event():
            try:
                return torch.cuda.Event(enable_timing=True, external=True)
            except TypeError:
                return torch.cuda.Event(enable_timing=True)

        def __enter__(self):
            if self.ev is not None:
                self.s = self._event()
                self.s.record()

        def __exit__(self, *exc):
            if self.ev is not None:
                e = self._event()
                e.record()
                self.ev.append((self.label, self.s, e))

    def _timed(self, label):
        return MoELayer._Timer(getattr(self, "_ev", None), label)

    def _fp8_experts(self, b: StepBuffers, tc: bool = False):
        """Expert batches: MXFP4 -> FP8 workspace conversion on a side stream,
        ring of `fp8_ring` batches, matmuls of batch i after its conversion.
        tc: the block-scaled FP8 tensor-core matmuls (MXFP8 token rows, E4M3
        workspace weights; FC1 writes h as MXFP8), else the CUDA-core GEMV."""
        E, H, I = self.E, self.H, self.I
        main = torch.cuda.current_stream(self.device)
        conv = self.conv_stream
        nb = len(self.batch_experts)
        converted = [torch.cuda.Event() for _ in range(nb)]
        consumed = [torch.cuda.Event() for _ in range(nb)]
        conv.wait_stream(main)  # routing / grouping done before the first matmul needs it

        def convert(i):
            if i >= self.ring:
                conv.wait_event(consumed[i - self.ring])  # ring slot free again
            L.mxfp4_to_fp8_ws(self.q1, self.e1, self.batch_experts[i], 2 * I, H, self.ws1, self.batch_slots[i],
                              dev_err=b.dev_err, stream=conv)
            L.mxfp4_to_fp8_ws(self.q2, self.e2, self.batch_experts[i], H, I, self.ws2, self.batch_slots[i],
                              dev_err=b.dev_err, stream=conv)
            converted[i].record(conv)

        for i in range(min(self.ring, nb)):
            convert(i)  # nothing to overlap yet: the whole GPU
        # the later conversions on reserved SMs beside the matmuls (the
        # setting is read when each call launches, also under graph capture)
        prev = L.moe_set_side_sms(self.side_sms) if tc and self.side_sms > 0 else None
        try:
            self._fp8_ring(b, tc, nb, convert, converted, consumed, main)
        finally:
            if prev is not None:
                L.moe_set_side_sms(prev)
        main.wait_stream(conv)

    def _fp8_ring(self, b, tc, nb, convert, converted, consumed, main):
        E, H, I = self.E, self.H, self.I
        for i in range(nb):
            e0 = i * self.batch
            e1 = min(E, e0 + self.batch)
            main.wait_event(converted[i])
            if tc:
                with self._timed("fp8_fc1_gemm"):
                    L.moe_mxfp4_mm(L.STAGE_FC1_SWIGLU, b.x_perm, L.FMT_MXFP8, b.offsets, E, I, H, b.h,
                                   L.FMT_MXFP8, fp8_ws=self.ws1, ws_slot_of_expert=self.ws_slot,
                                   act_scale=b.x_perm_scale, out_scale=b.h_scale,
                                   expert_begin=e0, expert_end=e1, mode=L.MODE_GEMM, dev_err=b.dev_err)
                with self._timed("fp8_fc2_gemm"):
                    L.moe_mxfp4_mm(L.STAGE_FC2, b.h, L.FMT_MXFP8, b.offsets, E, H, I, b.y, L.FMT_BF16,
                                   fp8_ws=self.ws2, ws_slot_of_expert=self.ws_slot, act_scale=b.h_scale,
                                   expert_begin=e0, expert_end=e1, mode=L.MODE_GEMM, dev_err=b.dev_err)
            else:
                with self._timed("fp8_fc1"):
                    L.moe_mxfp4_mm(L.STAGE_FC1_SWIGLU, b.x_perm, L.FMT_MXFP8, b.offsets, E, I, H, b.h,
                                   L.FMT_MXFP8, fp8_ws=self.ws1, ws_slot_of_expert=self.ws_slot,
                                   act_scale=b.x_perm_scale, expert_begin=e0, expert_end=e1, out_scale=b.h_scale,
                                   mode=self.mode, dev_err=b.dev_err)
                with self._timed("fp8_fc2"):
                    L.moe_mxfp4_mm(L.STAGE_FC2, b.h, L.FMT_MXFP8, b.offsets, E, H, I, b.y, L.FMT_BF16,
                                   fp8_ws=self.ws2, ws_slot_of_expert=self.ws_slot, act_scale=b.h_scale,
                                   expert_begin=e0, expert_end=e1, mode=self.mode, dev_err=b.dev_err)
            consumed[i].record(main)
            if i + self.ring < nb:
                convert(i + self.ring)

    # ------------------------------------------------------------ delta cache
    def attach_store(self, store, decay_shift: int = 31):
        """Manage the FP4 delta cache of a mixed layer on the device: ``store``
        holds the MXFP4 weights of every expert (q1, s1, q2, s2 stacked over
        E; device tensors, or pinned host tensors read over the CPU-GPU
        link).  ``update_cache`` then re-selects the cached experts from the
        running routing counts and copies newly promoted experts into their
        slots (moe_cache_select + moe_cache_fill), with no host sync."""
        assert self.fmt == "mixed"
        E, S = self.E, self.q1.shape[0]
        self.store = list(store)
        self.store_bytes = [t[0].numel() * t.element_size() for t in self.store]
        self.decay_shift = decay_shift
        self.counts = torch.zeros(E, dtype=torch.int32, device=self.device)
        es = self.expert_slot.cpu().numpy()
        se = np.full(S, -1, dtype=np.int32)
        for e in np.nonzero(es >= 0)[0]:
            se[es[e]] = e
        self.slot_expert = _dev(se, self.device)
        self.promoted = torch.empty(S, dtype=torch.int32, device=self.device)

    def update_cache(self, b: StepBuffers):
        """After a step: counts from the step's grouping, new cached set and
        slot maps, copies of the promoted experts (stream-ordered)."""
        L.moe_cache_select(b.offsets, self.counts, self.decay_shift, self.expert_slot, self.slot_expert,
                           self.promoted, dev_err=b.dev_err)
        L.moe_cache_fill(self.promoted, self.store, [self.q1, self.e1, self.q2, self.e2], self.store_bytes)

    def touched_weight_bytes(self, offsets: np.ndarray) -> int:
        """Bytes of packed weights (codes/nibbles + scales) of the experts the
        step touches: the decode roofline's algorithmic traffic."""
        cnt = np.diff(np.asarray(offsets))
        H, I = self.H, self.I
        w2_bytes = 3 * H * I // 4 + 3 * H * I // 32 * 2
        mx_bytes = 3 * H * I // 2 + 3 * H * I // 32
        tot = 0
        slot = None if self.expert_slot is None else self.expert_slot.cpu().numpy()
        for e in np.nonzero(cnt)[0]:
            if self.fmt == "w2" or (self.fmt == "mixed" and slot[e] < 0):
                tot += w2_bytes
            else:
                tot += mx_bytes
        return tot


class LayerGraph:
    """A captured layer step: ``run(x, logits)`` copies the step's inputs into
    the graph's own input buffers (stream-ordered device copies) and replays
    the graph; the output is ``out`` (overwritten by every run).  Inputs may
    be device tensors or pinned host tensors.  The buffers and weights the
    step uses stay owned by the graph and its layer."""

    def __init__(self, layer: MoELayer, T: int):
        dev = layer.device
        self.layer = layer
        self.x = torch.zeros((T, layer.H), dtype=torch.int16, device=dev)
        self.logits = torch.zeros((T, layer.E), dtype=torch.float32, device=dev)
        self.bufs = layer.buffers(T)
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):   # warm once outside the capture (library set-up, smem limits)
            layer.step(self.x, self.logits, self.bufs)
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.out = layer.step(self.x, self.logits, self.bufs)
        torch.cuda.synchronize(dev)

    def run(self, x: torch.Tensor, logits: torch.Tensor) -> torch.Tensor:
        self.x.copy_(x, non_blocking=True)
        self.logits.copy_(logits, non_blocking=True)
        self.graph.replay()
        return self.out
