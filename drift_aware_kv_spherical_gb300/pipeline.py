"""One drift-refresh step over all layers of a workload, through libpolestar.

A step runs, for every layer: spherical k-means (warm-started from the
previous step's centroids, or k-means++ when the window is built), NVFP4
residuals, proxy attention + KL drift against the previous step's
distribution, top-k drifting clusters and the sparse K/V refresh; then one
commit over the current block with the last layer's drift.  All buffers are
allocated once here (caller-side), so a step allocates nothing and can be
captured in a CUDA graph.

With offload=True (bf16 workloads) each layer's NVFP4 residuals are also
written, grouped by cluster, into a store in pinned host memory mapped into
the GPU, and the refresh takes the rows of the selected clusters as
reconstructed from that store (h~ = rho mu + deq(r)) instead of H
[Polestar §2.C, CPU offloading].

decode_step()/decode() run the step under the refresh schedule
(ps_schedule_step, [Polestar §2.A, schedule]): the drift path and the refresh
run only on steps the schedule marks, a full step refreshes every window
position from H, a new block resets the commit state and re-seeds k-means;
the commit runs every step on the last drift computed, and suffix-block
tokens commit only where the last layer's top-k position mask selects them
[Polestar §2.B, suffix block commitment].

scorer selects the drift signal: the proxy's fused KL (default), or one of
the ablation signals (cosine dissimilarity, entropy) computed by
ps_drift_score over the same proxy distributions [Polestar §4, ablation
studies].
"""

import torch

from . import polestar as ps
from . import workloads as wl


class LayerState:
    def __init__(self, w, device):
        B, N, C, d = w.B, w.N, w.C, w.d
        f32 = dict(dtype=torch.float32, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        u8 = dict(dtype=torch.uint8, device=device)
        dt = wl.torch_dtype(w)
        self.mu = torch.zeros(B, C, d, **f32)
        self.chat = torch.zeros(B, C, d, **f32)
        self.assign = torch.zeros(B, N, **i32)
        self.rho = torch.zeros(B, N, **f32)
        self.counts = torch.zeros(B, C, **i32)
        self.obj = torch.zeros(B, w.iters + 1, **f32)
        self.codes = torch.zeros(B, N, d // 2, **u8)
        self.scales = torch.zeros(B, N, d // 16, **u8)
        self.S = torch.zeros(B, **f32)
        self.A = [torch.zeros(B, N, C, **f32), torch.zeros(B, N, C, **f32)]
        self.D = torch.zeros(B, N, **f32)
        self.sel = torch.zeros(B, w.k, **i32)
        self.sel_score = torch.zeros(B, w.k, **f32)
        self.pos = torch.zeros(B, N, **i32)
        self.npos = torch.zeros(B, **i32)
        self.posmask = torch.zeros(B, N, **u8)
        self.Kc = torch.zeros(B, w.Ncache, w.Hkv, w.dh, dtype=dt, device=device)
        self.Vc = torch.zeros(B, w.Ncache, w.Hkv, w.dh, dtype=dt, device=device)


class Pipeline:
    """Buffers and the per-step call sequence for workload `w`."""

    def __init__(self, w, layers=None, device="cuda", offload=False, role=None,
                 scorer=ps.SCORER_KL):
        self.w = w
        self.scorer = scorer
        self.offload = offload
        if offload and w.dtype != "bf16":
            raise ValueError("the offload path reconstructs bf16 rows: bf16 workloads only")
        self.layers = w.layers if layers is None else layers
        self.device = device
        B, N, d, C = w.B, w.N, w.d, w.C
        sizes = dict(B=B, N=N, d=d, C=C, Hq=w.Hq, Hkv=w.Hkv, dh=w.dh, k=w.k, P=w.P,
                     V=w.V)
        self.ws = {op: ps.workspace(op, device=device, **sizes)
                   for op in (ps.OP_KMEANS, ps.OP_NVFP4, ps.OP_PROXY_KL, ps.OP_TOPK,
                              ps.OP_REFRESH, ps.OP_COMMIT)}
        self.state = [LayerState(w, device) for _ in range(self.layers)]
        if offload:
            rec = ps.ps_store_record_bytes(d)
            for st in self.state:
                st.store = ps.HostStore(B * N * rec)
                st.order = torch.zeros(B, N, dtype=torch.int32, device=device)
                st.cl_off = torch.zeros(B, C + 1, dtype=torch.int32, device=device)
                st.Ht = torch.zeros(B, N, d, dtype=torch.bfloat16, device=device)
        P = w.P
        self.role = (wl.make_roles(w) if role is None else role).to(device)
        self.all_pos = torch.arange(N, dtype=torch.int32, device=device).repeat(B, 1)
        self.all_npos = torch.full((B,), N, dtype=torch.int32, device=device)
        self._flags = None
        self._gin = None
        self._graphs = {}
        self.undecided = torch.ones(B, P, dtype=torch.uint8, device=device)
        self.d_sum = torch.zeros(B, P, dtype=torch.float32, device=device)
        self.d_cnt = torch.zeros(B, P, dtype=torch.int32, device=device)
        self.d_prev = torch.zeros(B, P, dtype=torch.float32, device=device)
        self.token = torch.zeros(B, P, dtype=torch.int32, device=device)
        self.conf = torch.zeros(B, P, dtype=torch.float32, device=device)
        self.commit = torch.zeros(B, P, dtype=torch.uint8, device=device)
        self.params = ps.CommitParams(w.tau_s, w.alpha, w.ratio, w.mode, 1)
        self.t = 0
        self._side = None
        self._after_proxy = None
        self.layer_done = []

    def side_streams(self):
        """Two streams for the ops off the critical path (NVFP4, commit)."""
        if self._side is None:
            self._side = [torch.cuda.Stream(self.device), torch.cuda.Stream(self.device)]
        return self._side

    def reset_block(self):
        self.undecided.fill_(1)
        self.d_sum.zero_()
        self.d_cnt.zero_()
        self.d_prev.zero_()

    def layer_step(self, l, H, Q, Wk, Wv, init_u=None, first=False, stream=None,
                   concurrent=False, joins=None, full=False):
        """One layer.  concurrent: the NVFP4 residuals run on a side stream
        (they depend on k-means only), and the event that ends them is
        appended to `joins` for the caller to wait on.  full: every window
        position is refreshed, from H (the top-k still sets the position
        mask)."""
        w, st = self.w, self.state[l]
        cur, prev = st.A[self.t % 2], st.A[(self.t + 1) % 2]
        ps.ps_kmeans_spherical(H, st.mu, st.assign, st.rho, st.chat, st.counts,
                               w.iters, init_mode=1 if first else 0, init_u=init_u,
                               objective=st.obj, ws=self.ws[ps.OP_KMEANS],
                               stream=stream)
        packed = None
        if concurrent:
            main = stream if stream is not None else torch.cuda.current_stream(self.device)
            side = self.side_streams()[0]
            side.wait_event(main.record_event())
            ps.ps_nvfp4_residual(H, st.mu, st.assign, st.rho, st.codes, st.scales, st.S,
                                 ws=self.ws[ps.OP_NVFP4], stream=side)
            if self.offload:
                ps.ps_nvfp4_pack_clusters(st.codes, st.scales, st.assign, w.C, st.store,
                                          st.order, st.cl_off, stream=side)
            packed = side.record_event()
            joins.append(packed)
        else:
            ps.ps_nvfp4_residual(H, st.mu, st.assign, st.rho, st.codes, st.scales, st.S,
                                 ws=self.ws[ps.OP_NVFP4], stream=stream)
            if self.offload:
                ps.ps_nvfp4_pack_clusters(st.codes, st.scales, st.assign, w.C, st.store,
                                          st.order, st.cl_off, stream=stream)
        fused = self.scorer == ps.SCORER_KL  # the proxy's own KL epilogue
        ps.ps_proxy_attn_kl(Q, st.chat, Wk, None if first or not fused else prev, cur, st.D,
                            w.Hkv, ws=self.ws[ps.OP_PROXY_KL], stream=stream)
        if not fused:  # an ablation signal over the same distributions
            ps.ps_drift_score(cur, None if first else prev, self.scorer, st.D, stream=stream)
        if concurrent:  # the drift is final here: the commit may start
            self._after_proxy = main.record_event()
        ps.ps_topk_drift(st.D, st.assign, st.counts, w.k, st.sel, st.sel_score, st.pos,
                         st.npos, st.posmask, ws=self.ws[ps.OP_TOPK], stream=stream)
        if full:
            if packed is not None:
                main.wait_event(packed)
            ps.ps_refresh_kv(H, self.all_pos, self.all_npos, Wk, Wv, st.Kc, st.Vc, w.Hkv, w.dh,
                             ws=self.ws[ps.OP_REFRESH], stream=stream)
            return
        src = H
        if self.offload:  # the selected clusters' rows, fetched from the host store
            if packed is not None:
                main.wait_event(packed)
            ps.ps_nvfp4_fetch_dequant(st.store, st.order, st.cl_off, st.sel, st.mu, st.rho,
                                      st.S, st.Ht, stream=stream)
            src = st.Ht
        ps.ps_refresh_kv(src, st.pos, st.npos, Wk, Wv, st.Kc, st.Vc, w.Hkv, w.dh,
                         ws=self.ws[ps.OP_REFRESH], stream=stream)

    def commit_step(self, logits, stream=None):
        w, last = self.w, self.state[-1]
        D_blk = last.D[:, w.blk_start:]
        suffix_sel = last.posmask[:, w.blk_start:]
        ps.ps_commit(logits, self.role, self.undecided, D_blk, w.N, self.d_sum,
                     self.d_cnt, self.d_prev, suffix_sel, w.N, self.params, self.token,
                     self.conf, self.commit, ws=self.ws[ps.OP_COMMIT], stream=stream)

    def step(self, Hs, Qs, Wks, Wvs, logits, init_us=None, first=False, stream=None,
             concurrent=False):
        """Hs/Qs/Wks/Wvs: per-layer tensors (lists of length `layers`).

        concurrent: the ops off the critical path (each layer's NVFP4
        residuals, the commit after the last layer's proxy) run on side
        streams joined back into `stream` before the step ends; the results
        are the same."""
        joins = []
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        for l in range(self.layers):
            self.layer_step(l, Hs[l], Qs[l], Wks[l], Wvs[l],
                            None if init_us is None else init_us[l], first, stream,
                            concurrent, joins)
        if concurrent:  # needs the last layer's drift only: overlaps its top-k and refresh
            side = self.side_streams()[1]
            side.wait_event(self._after_proxy)
            self.commit_step(logits, side)
            joins.append(side.record_event())
            for ev in joins:
                main.wait_event(ev)
        else:
            self.commit_step(logits, stream)
        self.t += 1


    def step_overlapped(self, Hs, Qs, Wks, Wvs, logits, main_stream, drift_stream,
                        forward=None, init_us=None, first=False):
        """The drift step hidden behind the caller's main forward on CUDA
        streams [Polestar §2.C, latency hiding]: clustering, quantisation,
        proxy attention and the update of the KV cache run on `drift_stream`
        while `main_stream` goes on with the model.

        forward(l, main_stream), if given, enqueues the caller's work that
        produces layer l's H and Q (l < layers) and, for l == layers, the
        block's logits.  Layer l's drift work forks from `main_stream` right
        after forward(l) -- it sees everything enqueued there up to that
        point -- and runs on `drift_stream` while forward(l + 1) runs on the
        main stream.  The commit forks after forward(layers).  At the end
        `main_stream` waits for `drift_stream`: the caches, the drift, the
        commit outputs and the state for the next step are ready for what
        the caller enqueues on `main_stream` next.  The event that ends
        layer l's drift work is kept in `self.layer_done[l]` for a caller
        that joins earlier, e.g. before a layer reads its cache.  The
        results are those of step() with the same inputs."""
        self.layer_done = []
        for l in range(self.layers):
            if forward is not None:
                forward(l, main_stream)
            drift_stream.wait_event(main_stream.record_event())
            self.layer_step(l, Hs[l], Qs[l], Wks[l], Wvs[l],
                            None if init_us is None else init_us[l], first, drift_stream)
            self.layer_done.append(drift_stream.record_event())
        if forward is not None:
            forward(self.layers, main_stream)
        drift_stream.wait_event(main_stream.record_event())
        self.commit_step(logits, drift_stream)
        self.t += 1
        main_stream.wait_event(drift_stream.record_event())

    def decode_step(self, act, Hs, Qs, Wks, Wvs, logits, init_us=None, stream=None):
        """One decode step under schedule actions `act` (ps.SCHED_* flags):
        SLIDE resets the block's commit state; REFRESH runs every layer's
        drift path (REINIT: k-means++ from init_us and no previous
        distribution; FULL: every position refreshed); the commit runs every
        step, on the last layer's most recent drift."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if act & ps.SCHED_SLIDE:
            with torch.cuda.stream(main):
                self.reset_block()
        if act & ps.SCHED_REFRESH:
            first = bool(act & ps.SCHED_REINIT)
            for l in range(self.layers):
                self.layer_step(l, Hs[l], Qs[l], Wks[l], Wvs[l],
                                None if init_us is None else init_us[l], first, stream,
                                full=bool(act & ps.SCHED_FULL))
            self.t += 1
        self.commit_step(logits, stream)

    def block_progress(self, stream=None):
        """(tokens committed by the last step, block decided) of the batch,
        read back to the host (one small copy and a wait on `stream`).  The
        batch decodes in lockstep: the count is the largest over its windows,
        and the block is decided when no window has an undecided
        current-block token."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if self._flags is None:  # pinned host memory the kernel writes straight into
            self._flags = ps.HostStore(16)
            self._flags_view = self._flags.view()[:8].view("int32")
        ps.ps_block_progress(self.commit, self.undecided, self.role, self._flags, stream=main)
        main.synchronize()
        return int(self._flags_view[0]), bool(self._flags_view[1])

    def graph_step(self, act, Hs, Qs, Wks, Wvs, logits, init_us=None, stream=None):
        """decode_step through CUDA graphs: the step's inputs are copied into
        fixed buffers, and the graph of (act, distribution parity) is
        captured on first use and replayed -- the same kernels in the same
        order as decode_step, without the host launching them one by one.
        The weights are captured by address and must not move between
        steps."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if self._gin is None:
            self._gin = dict(H=[h.clone() for h in Hs], Q=[q.clone() for q in Qs],
                             logits=logits.clone(),
                             u=None if init_us is None else [u.clone() for u in init_us],
                             W=[(wk.data_ptr(), wv.data_ptr()) for wk, wv in zip(Wks, Wvs)])
            self._graphs = {}
        g = self._gin
        if [(wk.data_ptr(), wv.data_ptr()) for wk, wv in zip(Wks, Wvs)] != g["W"]:
            raise ValueError("graph mode: the weights must stay at the same addresses")
        with torch.cuda.stream(main):
            for dst, src in zip(g["H"], Hs):
                dst.copy_(src, non_blocking=True)
            for dst, src in zip(g["Q"], Qs):
                dst.copy_(src, non_blocking=True)
            g["logits"].copy_(logits, non_blocking=True)
            if act & ps.SCHED_REINIT:
                for dst, src in zip(g["u"], init_us):
                    dst.copy_(src, non_blocking=True)
        key = (act, self.t % 2)
        if key not in self._graphs:
            t0 = self.t
            graph = torch.cuda.CUDAGraph()
            main.synchronize()
            with torch.cuda.graph(graph, capture_error_mode="relaxed"):
                self.decode_step(act, g["H"], g["Q"], Wks, Wvs, g["logits"], g["u"])
            self.t = t0  # capturing ran no kernel: the step happens at the replay
            self._graphs[key] = graph
            main.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(main):
            self._graphs[key].replay()
        if act & ps.SCHED_REFRESH:
            self.t += 1

    def decode(self, schedule, inputs, steps, stream=None, on_step=None, graphs=False):
        """Run `steps` decode steps under `schedule` (a ps.Schedule).

        inputs(t, block_start) returns (Hs, Qs, Wks, Wvs, logits, init_us) of
        step t, block_start being the schedule's current block; the first
        step builds the window (k-means++, full refresh).  on_step(t, act) is
        called after each step's work is enqueued.  graphs: run the steps
        through graph_step (the first step, which initialises the library's
        kernels, eagerly).  Returns the actions taken, one per step."""
        acts = []
        act = ps.SCHED_REFRESH | ps.SCHED_FULL | ps.SCHED_REINIT
        for t in range(steps):
            Hs, Qs, Wks, Wvs, logits, init_us = inputs(t, schedule.state.block_start)
            if graphs and t > 0:
                self.graph_step(act, Hs, Qs, Wks, Wvs, logits, init_us, stream)
            else:
                self.decode_step(act, Hs, Qs, Wks, Wvs, logits, init_us, stream)
            acts.append(act)
            if on_step is not None:
                on_step(t, act)
            committed, done = self.block_progress(stream)
            act = schedule.step(committed, done)
        return acts
