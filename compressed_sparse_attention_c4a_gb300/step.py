"""One layer step over resident device caches: the C-ABI calls in the order the layer runs them.

[P2] "DeepSeek V4 稀疏注意力完全解剖", 全景图 steps C-E: compress -> RMSNorm -> RoPE -> insert and SWA
insertion; indexer scores -> top-K; main attention over top-K entries plus the window; inverse RoPE.
This module owns output buffers and calls libdsa; it computes nothing itself.
"""
import math

import torch

from . import dsa

SM_SCALE = 1.0 / math.sqrt(512.0)
ROPE_THETA = 10000.0


def _query_group(spec, idx_heads):
    """Largest power of two <= 256/heads that divides every request's query count (1 for decode)."""
    if spec.queries != "all":
        return 1
    g = max(1, 256 // idx_heads)
    while g > 1 and any(n % g for n in spec.new):
        g //= 2
    return g


class LayerStep:
    """Device-resident state and buffers of one case (a dict from ``synth.make_case`` on cuda)."""

    def __init__(self, case, counted_topk=False, two_streams=False, dynamic_split=False, fused_select=False):
        spec = case["spec"]
        self.case, self.spec = case, spec
        dev = case["q"].device
        self.kind = spec.kind
        epb = case["epb"]
        self.main = dsa.pool(case["main_data"], epb, case["main_scale"])
        self.main_bt = dsa.block_table(case["bt_main"])
        self.swa = dsa.pool(case["swa_data"], 256, case["swa_scale"])
        self.swa_bt = dsa.block_table(case["bt_swa"])
        self.rope_main = dsa.rope(spec.rope_dim, ROPE_THETA)
        self.has_index = spec.idx_heads > 0
        self.fused_topk = False
        nq = case["nq"]
        if self.has_index:
            self.idx = dsa.pool(case["idx_data"], 64, case["idx_scale"], fmt=spec.idx_dtype)
            self.idx_bt = dsa.block_table(case["bt_idx"])
            self.rope_idx = dsa.rope(min(spec.rope_dim, spec.idx_dim), ROPE_THETA)
            self.ld = case["ld"]
            self.scores = torch.empty((nq, self.ld), dtype=torch.float32, device=dev)
            self.n_visible = torch.empty((nq,), dtype=torch.int32, device=dev)
            self.topk = torch.empty((nq, spec.topk), dtype=torch.int32, device=dev)
            self.q_group = _query_group(spec, spec.idx_heads)
            # counted_topk: the indexer counts the top-k's first radix digit while scoring and the top-k starts
            # from those counts (rows of up to 16,384 entries); off by default: on the decode batch the plain
            # indexer and top-k measure faster (the counts' key-prefix buckets are coarser than the plain top-k's
            # value buckets)
            self.fused_topk = counted_topk and self.ld <= 16384
            self.topk_ws = None
            if self.fused_topk:
                self.topk_ws = torch.zeros((dsa.dsa_index_topk_workspace_size(nq) // 4,), dtype=torch.int32, device=dev)
            # this step's compressor starts each request at start_pos: the indexer scores the key pages of
            # entries complete before it while the compressor still runs
            self.fresh_pos = case["start_pos"] if spec.index_compress else None
            # the indexer's work counter (CTAs take runs of items from it; it is left zero after each call)
            self.idx_work = torch.zeros((4,), dtype=torch.int32, device=dev)
        self.out = torch.empty((nq, spec.heads, spec.dim), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((nq, spec.heads), dtype=torch.float32, device=dev)
        max_keys = (spec.topk if self.has_index else case["bt_main"].shape[1] * epb) + spec.window
        ws = dsa.dsa_attn_workspace_size(nq, spec.heads, max_keys)
        self.attn_plan = dsa.dsa_attn_plan(nq, spec.heads, max_keys, spec.main_dtype)
        self.workspace = torch.empty((max(ws, 256),), dtype=torch.uint8, device=dev) if ws else None
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.max_new = max(spec.new) if spec.new else 0
        self.jobs = None
        self.two_streams = two_streams
        # dynamic_split: the indexer's CTAs take part of their work from a counter (idx_work) instead of an equal
        # static share; off by default (measured slower on the decode batch: more query-group switches)
        self.dynamic_split = dynamic_split
        self.side = None
        # fused_select: decode rows take the top-k and the attention in one call (one kernel when one cluster of
        # four CTAs per row holds all 64 heads, rows of at most 16,384 scores and k <= 512); off by default: on
        # the decode batch it measures level with the two launches (41.75 against 41.86 us a step; 38.1 against
        # 38.8 us with e2m1 indexer keys), its top-k phase running slower inside the attention kernel than the
        # top-k kernel alone
        self.fused_select = fused_select and self.has_index and spec.queries == "last" and not self.fused_topk
        self.select_attend_kernels = 2
        if self.fused_select:
            one = (tuple(self.attn_plan) == (64, 4, 1, 1) and spec.heads == 64 and self.ld <= 16384
                   and spec.topk <= 512)
            self.select_attend_kernels = 1 if one else 1 + self.attn_plan[3]

    # ---- stages ------------------------------------------------------------------------
    def _jobs(self):
        if self.jobs is None:
            c, pc = self.case, self.spec.gate == "channel"
            self.jobs = [dsa.compress_job(c["x_new"], c["z_new"], c["state_x"], c["state_z"], self.rope_main,
                                          self.main, self.main_bt, self.swa, self.swa_bt, per_channel=pc)]
            if self.has_index:
                self.jobs.append(dsa.compress_job(c["xi_new"], c["zi_new"], c["state_xi"], c["state_zi"],
                                                  self.rope_idx, self.idx, self.idx_bt, per_channel=pc))
        return self.jobs

    def compress_main(self):
        """Main-cache compressor + SWA insert."""
        c = self.case
        if self.spec.gate == "channel":  # the one-cache call takes a scalar gate only
            dsa.dsa_compress_jobs(self.kind, c["cu_new"], c["start_pos"], self.max_new, c["state_slot"],
                                  c["state_x"].shape[0], self._jobs()[:1], dev_status=self.status)
            return
        dsa.dsa_compress(self.kind, c["cu_new"], c["start_pos"], self.max_new, c["x_new"], c["z_new"], c["state_x"],
                         c["state_z"], c["state_slot"], self.rope_main, self.main, self.main_bt, self.swa,
                         self.swa_bt, dev_status=self.status)

    def compress_index(self):
        """Indexer-cache compressor (e4m3 or e2m1 keys + scale)."""
        c = self.case
        if self.has_index and self.spec.index_compress and self.spec.gate == "channel":
            dsa.dsa_compress_jobs(self.kind, c["cu_new"], c["start_pos"], self.max_new, c["state_slot"],
                                  c["state_x"].shape[0], self._jobs()[1:], dev_status=self.status)
        elif self.has_index and self.spec.index_compress:
            dsa.dsa_compress(self.kind, c["cu_new"], c["start_pos"], self.max_new, c["xi_new"], c["zi_new"],
                             c["state_xi"], c["state_zi"], c["state_slot"], self.rope_idx, self.idx, self.idx_bt,
                             dev_status=self.status)

    def compress(self):
        """Both compressors of the layer in one launch (main cache + SWA insert, and the indexer cache)."""
        c = self.case
        if not (self.has_index and self.spec.index_compress):
            self.compress_main()
            return
        dsa.dsa_compress_jobs(self.kind, c["cu_new"], c["start_pos"], self.max_new, c["state_slot"],
                              c["state_x"].shape[0], self._jobs(), dev_status=self.status)

    def index(self):
        """Indexer scores (counting each row's first top-k digit when the counted top-k follows)."""
        c = self.case
        if self.fused_topk:
            dsa.dsa_index_scores_counted(c["q8"], c["q_scale"], c["w"], c["q_pos"], c["q_req"], self.q_group,
                                         self.idx, self.idx_bt, self.scores, self.topk_ws, self.n_visible,
                                         dev_status=self.status, fresh_pos=self.fresh_pos,
                                         work=self.idx_work if self.dynamic_split else None)
        else:
            dsa.dsa_index_scores(c["q8"], c["q_scale"], c["w"], c["q_pos"], c["q_req"], self.q_group, self.idx,
                                 self.idx_bt, self.scores, self.n_visible, dev_status=self.status,
                                 fresh_pos=self.fresh_pos, work=self.idx_work if self.dynamic_split else None)

    def select(self):
        """Top-k of every query row (from the indexer's counts when it made them)."""
        if self.fused_topk:
            dsa.dsa_topk_counted(self.scores, self.n_visible, self.spec.topk, self.topk, self.topk_ws,
                                 dev_status=self.status)
        else:
            dsa.dsa_topk(self.scores, self.n_visible, self.spec.topk, self.topk, dev_status=self.status)

    def attend(self, topk=None):
        c, s = self.case, self.spec
        tk = (self.topk if topk is None else topk) if self.has_index else None
        k = s.topk if self.has_index else 0
        if s.queries == "last":
            dsa.dsa_sparse_attn_decode(c["q"], c["q_pos"], self.kind, tk, k, self.main, self.main_bt, self.swa,
                                       self.swa_bt, s.window, SM_SCALE, self.rope_main, self.out, self.lse,
                                       self.workspace, dev_status=self.status)
        else:
            dsa.dsa_sparse_attn_prefill(c["q"], c["q_pos"], c["q_req"], self.kind, tk, k, self.main, self.main_bt,
                                        self.swa, self.swa_bt, s.window, SM_SCALE, self.rope_main, self.out,
                                        self.lse, self.workspace, dev_status=self.status)

    def select_attend(self):
        """Top-k and attention in one call (decode rows): the top-k indices land in self.topk as well."""
        c, s = self.case, self.spec
        dsa.dsa_topk_sparse_attn_decode(c["q"], c["q_pos"], self.kind, self.scores, self.n_visible, s.topk, self.topk,
                                        self.main, self.main_bt, self.swa, self.swa_bt, s.window, SM_SCALE,
                                        self.rope_main, self.out, self.lse, self.workspace, dev_status=self.status)

    def launches_per_step(self):
        """Kernels one ``run()`` launches (compress: +1 ring kernel when a request appends > 1 token;
        attention: +1 merge kernel when a row's keys are split over several clusters)."""
        per_compress = 1 + (1 if self.max_new > 1 else 0)
        n = per_compress
        if self.has_index:
            n += (per_compress if self.spec.index_compress and self.two_streams else 0) + 1
            if self.fused_select and not self.two_streams:
                return n + self.select_attend_kernels
            n += 1
        n += self.attn_plan[3]
        return n

    def run(self):
        """The whole step: compress (+SWA insert), index, top-k, attention with inverse RoPE.

        One stream: both compressors in one launch, then the indexer, the top-k and the attention, each
        launched programmatically so that its set-up overlaps the tail of the kernel before it.  With
        ``two_streams`` the main-cache compressor and SWA insert run on a side stream beside the indexer chain
        (indexer compressor -> scores -> top-k) and the attention waits for both (a fork/join in a graph).
        """
        if not self.has_index:
            self.compress_main()
            self.attend()
            return self.out
        if not self.two_streams:
            self.compress()
            self.index()
            if self.fused_select:
                self.select_attend()
            else:
                self.select()
                self.attend()
            return self.out
        cur = torch.cuda.current_stream()
        if self.side is None:
            self.side = torch.cuda.Stream(device=cur.device)
        self.side.wait_stream(cur)
        with torch.cuda.stream(self.side):
            self.compress_main()
        self.compress_index()
        self.index()
        self.select()
        cur.wait_stream(self.side)
        self.attend()
        return self.out
