"""Device-resident synthetic model and the decode-stack driver.

DeviceModel draws every weight of a configuration on the GPU with the seeded
generator (synth.py / csrc/synth.cu), packs experts into per-expert blobs and
head matrices into records through the C ABI, and keeps descriptors for the
four calls.  DecodeStack runs decode steps of the layer stack through those
four calls (or, from step 1, through one of the two whole-step entries) and
can capture one step as a CUDA graph.  Around it: BatchedLayer (one layer
over T tokens), HostTierStack (routed experts in pinned host memory, gathered
into HBM a token ahead), merged_expert_blob / lora_merge_retention (the
adapter merged into the int4 weights, and how much of it survives) and
prediction_agreement (predicted routes against the layers' own routers).

Stack semantics (one decode step at token t; x_0 is the step's input):
  layer 0 routes with its own router (a head with H = 0) on x_0;
  layer N >= 1 uses the route head N-1 predicted at t-1 (at t = 0, when no
  prediction exists yet, its own router);
  y = experts(x_N); out_N = stream_N + combine(y); x_{N+1} = rms(out_N);
  head N runs on x_N with cur = layer N's route at t and prev = layer N's
  route at t-1 and predicts layer N+1's route for t+1.
A single-layer stack whose head predicts its own next route (self_predict)
routes with the head's prediction from step 1 on.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import moe, synth
from .configs import MoEConfig


def _align(n: int, a: int = 256) -> int:
    return (n + a - 1) // a * a


def _u16(shape, device):
    return torch.empty(shape, dtype=torch.int16, device=device)


class DeviceModel:
    def __init__(self, cfg: MoEConfig, device="cuda", heads: bool = True):
        self.cfg = cfg
        self.device = torch.device(device)
        self.blob_bytes = moe.moe_pool_expert_bytes(cfg.d, cfg.F, cfg.bits, cfg.group)
        if self.blob_bytes == 0:
            raise ValueError(f"unsupported expert shape {cfg}")
        self.stride = _align(self.blob_bytes)
        self.layers = []
        self._build(heads)

    # -------------------------------------------------------------- tensors
    def _affine_packed(self, tg: int, rows: int, cols: int, bits: int, sigma: float):
        dev = self.device
        q = torch.empty((rows, cols * bits // 32), dtype=torch.int32, device=dev)
        s = _u16((rows, cols // 64), dev)
        b = _u16((rows, cols // 64), dev)
        synth.gpu_affine(self.cfg.seed, tg, rows, cols, bits, sigma, q, s, b)
        out = torch.empty(_align(moe.moe_packed_matrix_bytes(rows, cols, bits)),
                          dtype=torch.uint8, device=dev)
        moe.moe_pack_matrix(q, s, b, rows, cols, bits, out)
        return out

    def _head_matrix(self, tg: int, rows: int, cols: int):
        c = self.cfg
        if c.head_prec == "fp16":
            return synth.gpu_gauss(c.seed, tg, _u16((rows, cols), self.device), c.sigma_w)
        return self._affine_packed(tg, rows, cols, 4, c.sigma_w)

    def _f16(self, tg: int, shape, sigma: float):
        return synth.gpu_gauss(self.cfg.seed, tg, _u16(shape, self.device), sigma)

    def _pool(self, layer: int, experts: list[int]):
        """Blobs of the given experts, packed; returns a uint8 tensor."""
        c, dev = self.cfg, self.device
        n, d, F, bits = len(experts), c.d, c.F, c.bits
        gq = torch.empty((n, F, d * bits // 32), dtype=torch.int32, device=dev)
        uq = torch.empty_like(gq)
        dq = torch.empty((n, d, F * bits // 32), dtype=torch.int32, device=dev)
        gs, gb, us, ub = (_u16((n, F, d // 64), dev) for _ in range(4))
        ds, db = (_u16((n, d, F // 64), dev) for _ in range(2))
        for i, e in enumerate(experts):
            synth.gpu_affine(c.seed, synth.tag(synth.GATE, layer, e), F, d, bits, c.sigma_w,
                             gq[i], gs[i], gb[i])
            synth.gpu_affine(c.seed, synth.tag(synth.UP, layer, e), F, d, bits, c.sigma_w,
                             uq[i], us[i], ub[i])
            synth.gpu_affine(c.seed, synth.tag(synth.DOWN, layer, e), d, F, bits, c.sigma_w,
                             dq[i], ds[i], db[i])
        pool = torch.empty(n * self.stride, dtype=torch.uint8, device=dev)
        moe.moe_pack_experts(d, F, n, bits, gq, gs, gb, uq, us, ub, dq, ds, db, pool,
                             self.stride)
        return pool

    def _lora(self, layer: int, e: int, ka: int, kb: int, din: int, dout: int):
        c = self.cfg
        A = self._f16(synth.tag(ka, layer, e), (c.lora_r, din), c.sigma_lora)
        B = self._f16(synth.tag(kb, layer, e), (dout, c.lora_r), c.sigma_lora)
        return A, B

    # -------------------------------------------------------------- build
    def _build(self, heads: bool):
        c = self.cfg
        routers = []
        for r in range(c.L):
            routers.append(self._head_matrix(synth.tag(synth.ROUTER, r), c.E, c.d))
        for r in range(c.L):
            ly = dict(keep=[])
            ly["pool"] = self._pool(r, list(range(c.E)))
            ly["shared"] = self._pool(r, [synth.SHARED_EXPERT]) if c.shared else None
            ed = moe.ExpertsDesc()
            ed.d, ed.F, ed.E, ed.bits = c.d, c.F, c.E, c.bits
            ed.pool = ly["pool"].data_ptr()
            ed.expert_stride = self.stride
            ed.shared = ly["shared"].data_ptr() if c.shared else None
            if c.lora_r and c.lora_on == "routed_down":
                A = _u16((c.E, c.lora_r, c.F), self.device)
                B = _u16((c.E, c.d, c.lora_r), self.device)
                for e in range(c.E):
                    synth.gpu_gauss(c.seed, synth.tag(synth.LORA_DOWN_A, r, e), A[e], c.sigma_lora)
                    synth.gpu_gauss(c.seed, synth.tag(synth.LORA_DOWN_B, r, e), B[e], c.sigma_lora)
                ly["keep"] += [A, B]
                ed.lora[2] = moe.LoraDesc(c.lora_r, c.lora_scale, A.data_ptr(), B.data_ptr(),
                                          c.lora_r * c.F, c.d * c.lora_r)
            if c.lora_r and c.lora_on == "shared_all" and c.shared:
                S = synth.SHARED_EXPERT
                for i, (ka, kb, din, dout) in enumerate(
                        [(synth.LORA_GATE_A, synth.LORA_GATE_B, c.d, c.F),
                         (synth.LORA_UP_A, synth.LORA_UP_B, c.d, c.F),
                         (synth.LORA_DOWN_A, synth.LORA_DOWN_B, c.F, c.d)]):
                    A, B = self._lora(r, S, ka, kb, din, dout)
                    ly["keep"] += [A, B]
                    ed.shared_lora[i] = moe.LoraDesc(c.lora_r, c.lora_scale, A.data_ptr(),
                                                     B.data_ptr(), 0, 0)
            ly["experts_desc"] = ed
            prec = moe.MOE_PREC_FP16 if c.head_prec == "fp16" else moe.MOE_PREC_AFFINE4
            rd = moe.HeadDesc()
            rd.d, rd.E, rd.H, rd.prec = c.d, c.E, 0, prec
            rd.lx = routers[r].data_ptr()
            ly["router_desc"] = rd
            ly["router"] = routers[r]
            if heads:
                tgt = synth.head_target(c, r)
                hd = moe.HeadDesc()
                hd.d, hd.E, hd.H, hd.prec = c.d, c.E, c.H, prec
                t = dict(lx=routers[tgt],
                         l_tab=self._f16(synth.tag(synth.L_TAB, r), (2 * c.E, c.E), c.sigma_w),
                         bl=self._f16(synth.tag(synth.BL, r), (c.E,), c.sigma_bias))
                if c.H:
                    t.update(fc1x=self._head_matrix(synth.tag(synth.FC1X, r), c.H, c.d),
                             fc1_tab=self._f16(synth.tag(synth.FC1_TAB, r), (2 * c.E, c.H), c.sigma_w),
                             b1=self._f16(synth.tag(synth.B1, r), (c.H,), c.sigma_bias),
                             fc2=self._head_matrix(synth.tag(synth.FC2, r), c.E, c.H),
                             b2=self._f16(synth.tag(synth.B2, r), (c.E,), c.sigma_bias))
                for k, v in t.items():
                    setattr(hd, k, v.data_ptr())
                ly["head"] = t
                ly["head_desc"] = hd
            self.layers.append(ly)
        torch.cuda.current_stream().synchronize()

    # -------------------------------------------------------------- sizes
    def head_bytes_per_token(self) -> int:
        """Bytes one decode token reads in one head call (dense matrices,
        2K gathered table rows per table, biases)."""
        c = self.cfg
        if c.head_prec == "fp16":
            dense = 2 * (c.H * c.d + c.E * c.H + c.E * c.d)
        else:
            dense = (moe.moe_packed_matrix_bytes(c.H, c.d, 4) if c.H else 0) + \
                (moe.moe_packed_matrix_bytes(c.E, c.H, 4) if c.H else 0) + \
                moe.moe_packed_matrix_bytes(c.E, c.d, 4)
        tables = 2 * c.K * 2 * (c.H + c.E)
        return dense + tables + 2 * (c.H + 2 * c.E)


class DecodeStack:
    """Batch-1 decode over `depth` layers (resident layers cycled).

    fused=True runs steady-state steps (t >= 1) as one persistent kernel
    (moe_decode_step); fused="chain" as two kernels per layer chained by
    programmatic dependent launch (moe_decode_step_chain); step 0, where every
    layer routes with its own router, always runs through the four per-layer
    calls."""

    def __init__(self, model: DeviceModel, fused=False):
        self.m = model
        c = self.cfg = model.cfg
        dev = model.device
        D = c.depth
        f32 = dict(dtype=torch.float32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.xin = torch.zeros(c.d, **f32)             # the step's input x_0
        self.xs = torch.zeros((D + 1, c.d), **f32)     # x_N, layer inputs
        self.stream = torch.zeros(c.d, **f32)          # residual stream
        self.y = torch.zeros((c.slots, c.d), **f32)
        self.logits = torch.zeros((D, c.E), **f32)
        # three rotating route sets: used at t, predicted for t+1, used at t-1
        self.r_idx = torch.zeros((3, D, c.K), **i32)
        self.r_w = torch.zeros((3, D, c.K), **f32)
        self.r_margin = torch.zeros((3, D), **f32)
        ed = model.layers[0]["experts_desc"]
        self.ffn_ws = torch.empty(moe.moe_expert_ffn_workspace_bytes(ed, 1, c.K),
                                  dtype=torch.uint8, device=dev)
        hd = model.layers[0].get("head_desc", model.layers[0]["router_desc"])
        self.head_ws = torch.empty(max(256, moe.moe_prerouter_head_workspace_bytes(hd, 1)),
                                   dtype=torch.uint8, device=dev)
        self.t = 0
        self.graphs = {}
        self.fused = bool(fused)
        self.chain = False
        if fused:
            L = model.layers
            self._ed = (moe.ExpertsDesc * c.L)(*[ly["experts_desc"] for ly in L])
            self._rd = (moe.HeadDesc * c.L)(*[ly["router_desc"] for ly in L])
            has_heads = all("head_desc" in ly for ly in L)
            self._hd = (moe.HeadDesc * c.L)(*[ly["head_desc"] for ly in L]) if has_heads else None
            self.sd = moe.StackDesc(C.cast(self._ed, C.c_void_p), C.cast(self._rd, C.c_void_p),
                                    C.cast(self._hd, C.c_void_p) if has_heads else None,
                                    c.L, c.depth, c.K, int(c.self_predict), 0, 0, None)
            self.chain = fused == "chain"
            nbytes = (moe.moe_decode_step_chain_workspace_bytes(self.sd) if self.chain
                      else moe.moe_decode_step_workspace_bytes(self.sd))
            self.step_ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def _layer(self, N: int):
        return self.m.layers[N % self.cfg.L]

    def _route_own(self, N: int, use: int):
        c = self.cfg
        ly = self._layer(N)
        moe.moe_prerouter_head(ly["router_desc"], self.xs[N], None, None, c.K, 1,
                               self.logits[N], self.head_ws)
        moe.moe_topk_route(self.logits[N], 1, c.E, c.K, self.r_idx[use, N], self.r_w[use, N],
                           self.r_margin[use, N])

    def enqueue_fused_step(self, t: int, events=None):
        """Enqueue step t >= 1 as one moe_decode_step launch."""
        if events is not None:
            events[0].record()
        call = moe.moe_decode_step_chain if self.chain else moe.moe_decode_step
        call(self.sd, self.xin, self.stream, self.r_idx, self.r_w, self.r_margin, t, self.step_ws)
        if events is not None:
            events[1].record()

    def status(self) -> int:
        """Status word of the fused step's workspace (synchronises)."""
        return moe.moe_decode_step_status(self.step_ws)

    def enqueue_step(self, t: int, ffn_events=None):
        """Enqueue one decode step (input already in self.xin) for token t.
        ffn_events: optional per-layer (start, end) CUDA events recorded
        around each layer's expert FFN call."""
        c = self.cfg
        D = c.depth
        use, nxt, prv = t % 3, (t + 1) % 3, (t - 1) % 3
        self.xs[0].copy_(self.xin)
        self.stream.copy_(self.xin)
        for N in range(D):
            ly = self._layer(N)
            if self._own(N, t):
                self._route_own(N, use)
            if ffn_events is not None:
                ffn_events[N][0].record()
            moe.moe_expert_ffn_int4(ly["experts_desc"], self.xs[N], self.r_idx[use, N], 1, c.K,
                                    self.y, self.ffn_ws)
            if ffn_events is not None:
                ffn_events[N][1].record()
            self._layer_tail(N, t)

    def _own(self, N: int, t: int) -> bool:
        """Layer N routes with its own router at step t (layer 0 without
        self-prediction; every layer at t = 0)."""
        return (N == 0 and not self.cfg.self_predict) or t == 0

    def _layer_tail(self, N: int, t: int):
        """Combine + residual of layer N, then its head's prediction of the
        next route of layer N + 1 (or of itself when self-predicting)."""
        c = self.cfg
        D = c.depth
        use, nxt, prv = t % 3, (t + 1) % 3, (t - 1) % 3
        ly = self._layer(N)
        moe.moe_combine_residual(self.y, self.r_w[use, N], 1, c.K, c.shared, c.d,
                                 self.stream, self.stream, self.xs[N + 1])
        tgt = N + 1 if N + 1 < D else (0 if c.self_predict else -1)
        if tgt >= 0:
            prev = self.r_idx[prv, N] if t > 0 else None
            moe.moe_prerouter_head(ly["head_desc"], self.xs[N], self.r_idx[use, N], prev,
                                   c.K, 1, self.logits[N], self.head_ws)
            moe.moe_topk_route(self.logits[N], 1, c.E, c.K, self.r_idx[nxt, tgt],
                               self.r_w[nxt, tgt], self.r_margin[nxt, tgt])

    def step(self, x0: torch.Tensor):
        """Run step self.t eagerly (or through its captured graph)."""
        self.xin.copy_(x0)
        t = self.t
        g = self.graphs.get(t % 3) if t >= 1 else None
        if g is not None:
            g.replay()
        elif self.fused and t >= 1:
            self.enqueue_fused_step(t)
        else:
            self.enqueue_step(t)
        self.t += 1

    def capture(self):
        """Capture the steady-state step (t >= 1) once per route rotation."""
        for rot in range(3):
            t = rot if rot >= 1 else 3
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                if self.fused:
                    self.enqueue_fused_step(t)
                else:
                    self.enqueue_step(t)
            self.graphs[rot] = g

    def own_routes(self, t: int):
        """Right after step t (t >= 1, per-call path): the top-K of every
        layer's own router on the input x_N it had at t, with the logits'
        margins -- what the layer would have used without the prediction."""
        c = self.cfg
        assert not self.fused and t >= 1 and self.t == t + 1
        dev = self.m.device
        own = torch.empty((c.depth, c.K), dtype=torch.int32, device=dev)
        w = torch.empty((c.depth, c.K), dtype=torch.float32, device=dev)
        mg = torch.empty(c.depth, dtype=torch.float32, device=dev)
        z = torch.empty(c.E, dtype=torch.float32, device=dev)
        for N in range(c.depth):
            moe.moe_prerouter_head(self._layer(N)["router_desc"], self.xs[N], None, None, c.K, 1,
                                   z, self.head_ws)
            moe.moe_topk_route(z, 1, c.E, c.K, own[N], w[N], mg[N])
        return own, mg

    def used_routes(self, t: int):
        """(idx [depth][K], w, margin) the layers used at step t (valid right
        after step t, before step t+2 overwrites the rotation)."""
        u = t % 3
        return self.r_idx[u].clone(), self.r_w[u].clone(), self.r_margin[u].clone()


class HostTierStack(DecodeStack):
    """Per-call decode with the routed experts in pinned host memory.

    Every resident layer's routed pool is moved to pinned host memory (the
    shared expert stays in HBM).  At the start of step t the routes of every
    predicted layer are already known (made during step t - 1), so a side
    stream gathers each layer's K experts into that layer's HBM slots
    (moe_gather_experts, reading host memory over NVLink-C2C) while the main
    stream computes; layer N's expert call waits only for its own gather.  A
    layer that routes itself in the step gathers right after its router.
    Results are those of DecodeStack bit for bit (same kernels, same bytes)."""

    def __init__(self, model: DeviceModel):
        super().__init__(model)
        c = self.cfg
        if c.lora_r and c.lora_on == "routed_down":
            raise ValueError("routed-expert adapters are not gathered with the blobs")
        dev = model.device
        self.host_pools = []
        for ly in model.layers:
            h = torch.empty(ly["pool"].numel(), dtype=torch.uint8, pin_memory=True)
            h.copy_(ly["pool"])
            self.host_pools.append(h)
        self.blob = moe.moe_pool_expert_bytes(c.d, c.F, c.bits, 64)
        self.slots = torch.empty((c.depth, c.K * model.stride), dtype=torch.uint8, device=dev)
        self.slot_idx = torch.empty((c.depth, c.K), dtype=torch.int32, device=dev)
        self.eds = []
        for N in range(c.depth):
            e = moe.ExpertsDesc.from_buffer_copy(self._layer(N)["experts_desc"])
            e.pool = self.slots[N].data_ptr()
            e.E = c.K
            self.eds.append(e)
        self.side = torch.cuda.Stream(device=dev)
        self.ready = [torch.cuda.Event() for _ in range(c.depth)]

    def gather(self, N: int, t: int, stream=None):
        """Layer N's routed experts of step t, host pool -> its HBM slots."""
        c = self.cfg
        moe.moe_gather_experts(self.host_pools[N % c.L].data_ptr(), self.m.stride, c.E,
                               self.r_idx[t % 3, N], c.K, self.blob, self.slots[N],
                               self.m.stride, self.slot_idx[N], stream)

    def enqueue_step(self, t: int, ffn_events=None):
        c = self.cfg
        use = t % 3
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            for N in range(c.depth):
                if not self._own(N, t):
                    self.gather(N, t, self.side)
                    self.ready[N].record(self.side)
        self.xs[0].copy_(self.xin)
        self.stream.copy_(self.xin)
        for N in range(c.depth):
            if self._own(N, t):
                self._route_own(N, use)
                self.gather(N, t, main)
            else:
                main.wait_event(self.ready[N])
            if ffn_events is not None:
                ffn_events[N][0].record()
            moe.moe_expert_ffn_int4(self.eds[N], self.xs[N], self.slot_idx[N], 1, c.K, self.y,
                                    self.ffn_ws)
            if ffn_events is not None:
                ffn_events[N][1].record()
            self._layer_tail(N, t)
        main.wait_stream(self.side)


class HostTierChain(DecodeStack):
    """Chained decode steps (moe_decode_step_chain) with the routed experts in
    pinned host memory behind an HBM cache per layer.

    Every resident layer's routed pool is moved to pinned host memory (the
    shared expert stays in HBM).  Each layer of the stack gets its own cache
    of `cache_slots` expert slots in HBM (least recently used out,
    moe_cache_experts; its hit and miss counts in `stats`).  At the start of
    step t the routes of layers 1 .. depth-1 are already known (predicted
    during step t - 1), so a side stream runs every such layer's cache update
    -- the decision and the copies of its misses over NVLink-C2C -- while the
    main stream runs the chained step, whose layer N waits only for its own
    update (moe_stack_desc.layer_ready) and reads its experts from the cache
    slots (moe_stack_desc.slot_map); free_sms SMs can be left to the copies
    (moe_stack_desc.free_sms).  Layer 0 routes with its own router inside
    the step, so its experts stay resident in HBM.  Results are those of the
    HBM-resident chained step bit for bit (same kernels, same bytes)."""

    def __init__(self, model: DeviceModel, cache_slots: int, free_sms: int = 0, side_streams: int = 1):
        super().__init__(model, fused="chain")
        c = self.cfg
        if c.self_predict:
            raise ValueError("a self-predicting single layer has no layer routed a token ahead")
        if c.lora_r and c.lora_on == "routed_down":
            raise ValueError("routed-expert adapters are not cached with the blobs")
        dev = model.device
        D, K = c.depth, c.K
        self.C = cache_slots
        self.host_pools = []
        for ly in model.layers:
            h = torch.empty(ly["pool"].numel(), dtype=torch.uint8, pin_memory=True)
            h.copy_(ly["pool"])
            self.host_pools.append(h)
        # (the model's HBM pools stay allocated, for stacks that share the model;
        # this stack reads only layer 0's, the layer that routes itself)
        self.blob = moe.moe_pool_expert_bytes(c.d, c.F, c.bits, 64)
        i32 = dict(dtype=torch.int32, device=dev)
        self.cache = torch.empty((D, cache_slots * model.stride), dtype=torch.uint8, device=dev)
        self.tags = torch.full((D, cache_slots), -1, **i32)
        self.ages = torch.zeros((D, cache_slots), **i32)
        self.clock = torch.zeros(D, **i32)
        self.slot_map = torch.zeros((D, K), **i32)
        self.plan = torch.zeros((D, K), **i32)
        self.stats = torch.zeros((D, 2), **i32)
        # one descriptor per layer of the stack: layer 0 on its resident pool,
        # every other on its cache
        self._ed = (moe.ExpertsDesc * D)()
        self._rd = (moe.HeadDesc * D)()
        self._hd = (moe.HeadDesc * D)()
        for N in range(D):
            ly = self._layer(N)
            e = moe.ExpertsDesc.from_buffer_copy(ly["experts_desc"])
            if N > 0:
                e.pool = self.cache[N].data_ptr()
            self._ed[N] = e
            self._rd[N] = ly["router_desc"]
            self._hd[N] = ly["head_desc"]
        self.sd = moe.StackDesc(C.cast(self._ed, C.c_void_p), C.cast(self._rd, C.c_void_p),
                                C.cast(self._hd, C.c_void_p), D, D, K, 0, 0, 0, None)
        self.sd.slot_map = self.slot_map.data_ptr()
        self.sd.free_sms = free_sms             # SMs left to the cache copies
        self.step_ws = torch.zeros(moe.moe_decode_step_chain_workspace_bytes(self.sd),
                                   dtype=torch.uint8, device=dev)
        # the layers' updates go round-robin over side_streams streams (more
        # copies in flight over C2C at once)
        self.sides = [torch.cuda.Stream(device=dev) for _ in range(max(1, side_streams))]
        self.side = self.sides[0]
        self.ready = [torch.cuda.Event() for _ in range(D)]
        self._ready_ptrs = None

    def hit_rate(self) -> float:
        """Hits / (hits + misses) over every cache update so far."""
        h, m = self.stats.sum(0).tolist()
        return h / max(1, h + m)

    def update(self, N: int, t: int, stream):
        """Layer N's cache for the route of step t: hits kept, misses copied
        from host memory; slot_map[N] names each route position's slot."""
        c = self.cfg
        moe.moe_cache_experts(self.host_pools[N % c.L].data_ptr(), self.m.stride, c.E,
                              self.r_idx[t % 3, N], c.K, self.blob, self.cache[N], self.m.stride,
                              self.C, self.tags[N], self.ages[N], self.clock[N:N + 1],
                              self.slot_map[N], self.plan[N], self.stats[N], stream)

    def enqueue_fused_step(self, t: int, events=None, update_events=None):
        """Step t >= 1: the cache updates of layers 1 .. depth-1 on the side
        stream, the chained step on the current one (layer N after its
        update).  update_events: optional (start, [depth]) events -- start
        recorded on the current stream when the step begins, [N] on the side
        stream when layer N's update has finished."""
        c = self.cfg
        main = torch.cuda.current_stream()
        if update_events is not None:
            update_events[0].record(main)
        for sd in self.sides:
            sd.wait_stream(main)
        for N in range(1, c.depth):
            sd = self.sides[(N - 1) % len(self.sides)]
            with torch.cuda.stream(sd):
                self.update(N, t, sd)
                self.ready[N].record(sd)
                if update_events is not None:
                    update_events[1][N].record(sd)
        if self._ready_ptrs is None:         # event handles exist once recorded
            self._ready_ptrs = (C.c_void_p * c.depth)(
                *([None] + [C.c_void_p(e.cuda_event) for e in self.ready[1:]]))
            self.sd.layer_ready = C.cast(self._ready_ptrs, C.c_void_p)
        if events is not None:
            events[0].record()
        moe.moe_decode_step_chain(self.sd, self.xin, self.stream, self.r_idx, self.r_w,
                                  self.r_margin, t, self.step_ws)
        if events is not None:
            events[1].record()
        for sd in self.sides:
            main.wait_stream(sd)

    def enqueue_step(self, t: int, ffn_events=None):
        """Step 0 (every layer routes itself): the per-call path, each layer's
        cache updated right after its router."""
        c = self.cfg
        use = t % 3
        self.xs[0].copy_(self.xin)
        self.stream.copy_(self.xin)
        for N in range(c.depth):
            ly = self._layer(N)
            self._route_own(N, use)
            ed = ly["experts_desc"] if N == 0 else self._slot_desc(N)
            idx = self.r_idx[use, N]
            if N > 0:
                self.update(N, t, torch.cuda.current_stream())
                idx = self.slot_map[N]
            moe.moe_expert_ffn_int4(ed, self.xs[N], idx, 1, c.K, self.y, self.ffn_ws)
            self._layer_tail(N, t)

    def _slot_desc(self, N: int):
        """Layer N's cache as an expert pool of C experts (for the per-call
        expert FFN, which indexes it by slot)."""
        e = moe.ExpertsDesc.from_buffer_copy(self._ed[N])
        e.E = self.C
        return e


class BatchedLayer:
    """One MoE layer over T tokens at once (prefill, batched decode).

    Inputs: x (bf16 [T][d], the layer's normalised input), the residual
    stream (fp32 [T][d]), this layer's routes (cur_idx, cur_w: predicted by
    the previous layer's head) and the previous token's routes (prev_idx).
    One step enqueues, for all T tokens: the prerouter head and top-K that
    predict the next layer's routes, the expert FFN on the current routes
    (grouped by expert inside the call), and the combine + residual with the
    next layer's fp32 input."""

    def __init__(self, model: DeviceModel, T: int, layer: int = 0):
        self.m = model
        c = self.cfg = model.cfg
        dev = model.device
        self.T = T
        self.ly = model.layers[layer]
        f32 = dict(dtype=torch.float32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.x = torch.zeros((T, c.d), dtype=torch.bfloat16, device=dev)
        self.res = torch.zeros((T, c.d), **f32)
        self.out = torch.zeros((T, c.d), **f32)
        self.x_next = torch.zeros((T, c.d), **f32)
        self.cur_idx = torch.zeros((T, c.K), **i32)
        self.cur_w = torch.zeros((T, c.K), **f32)
        self.prev_idx = torch.zeros((T, c.K), **i32)
        self.next_idx = torch.zeros((T, c.K), **i32)
        self.next_w = torch.zeros((T, c.K), **f32)
        self.next_margin = torch.zeros(T, **f32)
        self.logits = torch.zeros((T, c.E), **f32)
        self.y = torch.zeros((T, c.slots, c.d), **f32)
        ed = self.ly["experts_desc"]
        self.ffn_ws = torch.empty(moe.moe_expert_ffn_workspace_bytes(ed, T, c.K),
                                  dtype=torch.uint8, device=dev)
        self.head_ws = torch.empty(max(256, moe.moe_prerouter_head_workspace_bytes(
            self.ly["head_desc"], T)), dtype=torch.uint8, device=dev)

    def route_own(self):
        """Routes for the current input from the layer's own router (for
        inputs that have no predicted route yet); prev = the previous token's
        route (token 0 takes its own)."""
        c = self.cfg
        moe.moe_prerouter_head(self.ly["router_desc"], self.x, None, None, c.K, self.T,
                               self.logits, self.head_ws)
        moe.moe_topk_route(self.logits, self.T, c.E, c.K, self.cur_idx, self.cur_w)
        self.prev_idx[1:].copy_(self.cur_idx[:-1])
        self.prev_idx[0].copy_(self.cur_idx[0])

    def enqueue(self, ffn_events=None):
        c, T = self.cfg, self.T
        moe.moe_prerouter_head(self.ly["head_desc"], self.x, self.cur_idx, self.prev_idx, c.K,
                               T, self.logits, self.head_ws)
        moe.moe_topk_route(self.logits, T, c.E, c.K, self.next_idx, self.next_w,
                           self.next_margin)
        if ffn_events is not None:
            ffn_events[0].record()
        moe.moe_expert_ffn_int4(self.ly["experts_desc"], self.x, self.cur_idx, T, c.K, self.y,
                                self.ffn_ws)
        if ffn_events is not None:
            ffn_events[1].record()
        moe.moe_combine_residual(self.y, self.cur_w, T, c.K, c.shared, c.d, self.res, self.out,
                                 self.x_next)


# ---------------------------------------------------------------- LoRA merge
def expert_sections(cfg: MoEConfig):
    """(byte offset, row stride, rows, cols) of the gate, up and down rows of
    one expert blob (gate row f = record 2f, up row f = record 2f + 1 of the
    gate/up section; the down section starts on the next 256-byte boundary)."""
    rec_d = moe.moe_record_bytes(cfg.d, cfg.bits)
    rec_f = moe.moe_record_bytes(cfg.F, cfg.bits)
    down = _align(2 * cfg.F * rec_d)
    return [(0, 2 * rec_d, cfg.F, cfg.d), (rec_d, 2 * rec_d, cfg.F, cfg.d),
            (down, rec_f, cfg.d, cfg.F)]


def merged_expert_blob(blob: torch.Tensor, cfg: MoEConfig, adapters) -> torch.Tensor:
    """A copy of one expert blob with its gate / up / down adapters (three
    LoraDesc, r == 0 for none) merged into the weights and requantised, on
    the GPU (moe_merge_lora)."""
    out = blob.clone()
    for (off, stride, rows, cols), l in zip(expert_sections(cfg), adapters):
        if l.r:
            moe.moe_merge_lora(blob.data_ptr() + off, stride, rows, cols, cfg.bits, l.A, l.B,
                               l.r, l.scale, out.data_ptr() + off, stride)
    return out


def lora_merge_retention(model: DeviceModel, layer: int = 0, T: int = 16, tag: int = 977) -> dict:
    """How much of the shared expert's LoRA delta survives merging it into
    the int4 weights: the shared slot's output y over T seeded tokens with
    the base weights (no adapter), the unfused adapter and the merged,
    requantised weights; retention = <y_m - y_b, y_l - y_b> / |y_l - y_b|^2
    and the merged result's error |y_m - y_l| / |y_l - y_b|."""
    c = model.cfg
    ly = model.layers[layer]
    ed = ly["experts_desc"]
    merged = merged_expert_blob(ly["shared"], c, [ed.shared_lora[i] for i in range(3)])

    def desc(shared: torch.Tensor, adapters: bool):
        e = moe.ExpertsDesc.from_buffer_copy(ed)
        e.shared = shared.data_ptr()
        if not adapters:
            for i in range(3):
                e.shared_lora[i] = moe.LoraDesc()
        return e

    x = torch.from_numpy(synth.gauss(c.seed, tag, (T, c.d), 1.0)).to(model.device)
    idx = torch.from_numpy(synth.routes(c.seed, tag + 1, T, c.E, c.K)).to(model.device)
    ys = []
    for e in (desc(ly["shared"], False), desc(ly["shared"], True), desc(merged, False)):
        y = torch.empty((T, c.K + 1, c.d), device=model.device)
        ws = torch.empty(moe.moe_expert_ffn_workspace_bytes(e, T, c.K), dtype=torch.uint8,
                         device=model.device)
        moe.moe_expert_ffn_int4(e, x, idx, T, c.K, y, ws)
        ys.append(y[:, c.K].double())
    yb, yl, ym = ys
    dl, dm = yl - yb, ym - yb
    n2 = float((dl * dl).sum())
    return {"retention": float((dm * dl).sum()) / n2,
            "merged_error": float(((ym - yl) ** 2).sum() / n2) ** 0.5,
            "delta_rms_over_y_rms": float((n2 / float((yl * yl).sum())) ** 0.5),
            "tokens": T, "layer": layer, "merged_blob": merged}


# ---------------------------------------------------------------- prediction agreement
def prediction_agreement(model: DeviceModel, steps: int = 16) -> dict:
    """How often the predicted route (head N-1 at t-1) agrees with the route
    layer N's own router would take on its input at t, over `steps` seeded
    decode steps (t = 1 .. steps, per-call path).  Layers that route
    themselves (layer 0 without self-prediction) are left out.  Returns the
    fraction of layer-steps whose K-sets are equal, the mean overlap
    |predicted & own| / K, and K / E, the overlap two independent uniform
    K-subsets have on average (random synthetic heads sit near it)."""
    c = model.cfg
    st = DecodeStack(model)
    first = 0 if c.self_predict else 1
    equal = overlap = n = 0
    for t in range(steps + 1):
        st.step(torch.from_numpy(synth.step_input(c, t)[0]).to(model.device))
        if t == 0:
            continue
        own, _ = st.own_routes(t)
        used, _, _ = st.used_routes(t)
        own, used = own.cpu().numpy(), used.cpu().numpy()
        for N in range(first, c.depth):
            a, b = set(own[N].tolist()), set(used[N].tolist())
            equal += int(a == b)
            overlap += len(a & b) / c.K
            n += 1
    return {"layer_steps": n, "equal_sets": equal / n, "mean_overlap": overlap / n,
            "chance_overlap": c.K / c.E, "steps": steps}
