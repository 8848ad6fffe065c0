"""Decode-step driver over libpkv: pool tensors, block tables and one decode step.

One decode step over a batch (all through the C ABI):

1. host, ``pkv_prepare_append``: one slot per sequence, new blocks at block
   boundaries, copy-on-write pairs for shared blocks;
2. the step's tables, lengths, slots and pairs go host -> device from pinned
   double-buffered staging (the host can prepare step k+1 while step k runs);
3. ``pkv_copy_blocks`` once for the step, across all layers;
4. per layer: the new token's K/V appended and attention over the cache
   including it -- one launch that appends and attends (the default for an fp16
   cache, and for an E4M3 cache whose batch gives each CTA at most four
   (sequence, head) pairs), or ``pkv_append`` then the attention started early
   behind it (an E4M3 cache with more). With the shared-prefix cascade (HND
   pools, head_dim 128, fp16 or E4M3, on by default), the host plans groups of
   sequences that share leading blocks (``pkv_cascade_plan``) and each layer
   first runs ``pkv_prefix_attention`` over the groups' prefixes, then
   ``pkv_decode_attention_ex`` over the private rest (with the append when
   fused).

The driver also replays a workload's set-up script (admissions, forks, dummy
churn, multi-token writes). It holds no arithmetic of the method: slots,
copies, tables and attention all come from the library.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

import workloads as wl

from . import binding as bd


# E4M3 cache: the attention launch appends the step's rows itself while each of its CTAs
# ends at most this many (sequence, head) pairs on average, else a separate append launch
FUSED_E4M3_UNITS_PER_CTA = 4


class DecodeEngine:
    def __init__(self, w: wl.Workload, device: str = "cuda", fill: str = "torch", max_new_per_step: int = 1,
                 fused: Optional[bool] = None, cascade: bool = True):
        self.w = w
        # append inside the attention launch (pkv_decode_append_attention). By default
        # always on an fp16 cache; on an E4M3 cache only while each CTA of the attention
        # launch ends few (sequence, head) pairs: each costs its producer warp a load-
        # quantise-store-fence chain, paid one after another by a CTA whose range holds
        # many short sequences, and past about four a CTA on average the separate append
        # launch wins (7B batch 32: 1.7 a CTA, fused +4 % per step; 13B batch 128: 8.4,
        # fused -9 %)
        if fused is None:
            fused = True
            if w.kv_dtype != "f16":
                grid = bd.decode_launch_info(w.num_seqs, w.head_dim, w.kv_dtype)["grid_ctas"]
                fused = w.num_seqs * w.num_heads <= FUSED_E4M3_UNITS_PER_CTA * grid
        self.fused = bool(fused)
        # shared-prefix cascade: where a prefix pass is built (fp16 and E4M3 pools, HND, head_dim 128)
        self.cascade = bool(cascade) and w.layout == "HND" and w.head_dim == 128
        self.device = torch.device(device)
        shape = wl.pool_shape(w)
        self.k_scale = self.v_scale = None
        if w.kv_dtype == "e4m3":
            if fill == "numpy":
                self.k_pool = torch.from_numpy(wl.pool_codes_e4m3(w, 0)).to(self.device)
                self.v_pool = torch.from_numpy(wl.pool_codes_e4m3(w, 1)).to(self.device)
                self.k_scale = torch.from_numpy(wl.pool_scales(w, 0)).to(self.device)
                self.v_scale = torch.from_numpy(wl.pool_scales(w, 1)).to(self.device)
            else:
                self.k_pool, self.k_scale = wl.torch_e4m3_pool(w, 0, self.device)
                self.v_pool, self.v_scale = wl.torch_e4m3_pool(w, 1, self.device)
        elif fill == "numpy":
            self.k_pool = torch.from_numpy(wl.pool_values(w, 0)).to(self.device)
            self.v_pool = torch.from_numpy(wl.pool_values(w, 1)).to(self.device)
        elif fill == "torch":
            self.k_pool = wl.torch_normal_fp16(w.seed, (100,), shape, self.device)
            self.v_pool = wl.torch_normal_fp16(w.seed, (101,), shape, self.device)
        else:
            raise ValueError(fill)
        self.pool = bd.Pool(w.num_layers, w.num_blocks, w.block_size, w.num_heads, w.head_dim, w.layout,
                            self.k_pool, self.v_pool, w.free_order, kv_dtype=w.kv_dtype, k_scale=self.k_scale,
                            v_scale=self.v_scale)
        S, maxb = w.num_seqs, w.max_blocks
        self.tables = np.full((S, maxb), -1, dtype=np.int32)
        self.lens = np.zeros(S, dtype=np.int32)
        self.dummies = {}
        self.tables_d = torch.full((S, maxb), -1, dtype=torch.int32, device=self.device)
        self.lens_d = torch.zeros(S, dtype=torch.int32, device=self.device)
        self.status = torch.zeros(4, dtype=torch.int32, device=self.device)
        self.workspace = bd.new_workspace(S, w.num_heads, w.head_dim, self.device)
        # the cascade plan on the device (refreshed with every step's tables) and the prefix pieces
        self.groups_d = torch.zeros((max(S, 1), 4), dtype=torch.int32, device=self.device)
        self.begin_d = torch.zeros(max(S, 1), dtype=torch.int32, device=self.device)
        self.pieces = (torch.empty(bd.prefix_pieces_bytes(S, w.num_heads, w.head_dim), dtype=torch.uint8,
                                   device=self.device) if self.cascade else None)
        self.plan_groups, self.plan_splits, self.plan_prefix = 0, 0, 0
        self.plan = np.zeros((0, 4), dtype=np.int32)
        self._cap_slots = S * max_new_per_step
        self.slots_d = torch.zeros(max(self._cap_slots, 1), dtype=torch.int64, device=self.device)
        self.pairs_d = torch.zeros((max(self._cap_slots, 1), 2), dtype=torch.int32, device=self.device)
        # pinned, double-buffered host staging for the per-step H2D copies
        self._stage = []
        for _ in range(2):
            self._stage.append({
                "tables": torch.empty((S, maxb), dtype=torch.int32).pin_memory(),
                "lens": torch.empty(S, dtype=torch.int32).pin_memory(),
                "slots": torch.empty(max(self._cap_slots, 1), dtype=torch.int64).pin_memory(),
                "pairs": torch.empty((max(self._cap_slots, 1), 2), dtype=torch.int32).pin_memory(),
                "groups": torch.zeros((max(S, 1), 4), dtype=torch.int32).pin_memory(),
                "begin": torch.zeros(max(S, 1), dtype=torch.int32).pin_memory(),
                "event": None,
            })
        self._buf = 0
        self.last_pairs = np.zeros((0, 2), dtype=np.int32)
        self.cow_log = []             # every copy-on-write pair array the script's writes produced
        self.last_slots = np.zeros(0, dtype=np.int64)

    # ------------------------------------------------------------------ set-up script
    def run_script(self, values: str = "numpy", stream=None):
        """Replay the workload's host operations; ``write`` ops append generated K/V through the kernels."""
        w, B = self.w, self.w.block_size
        for op_index, op in enumerate(w.script):
            kind = op[0]
            if kind == "admit":
                _, s, T = op
                nb = -(-T // B)
                ids = self.pool.alloc(nb)
                self.tables[s, :nb] = ids
                self.lens[s] = T
            elif kind == "fork":
                _, src, dst = op
                nb = -(-int(self.lens[src]) // B)
                self.pool.incref(self.tables[src, :nb])
                self.tables[dst] = self.tables[src]
                self.lens[dst] = self.lens[src]
            elif kind == "dummy_alloc":
                _, d, n = op
                self.dummies[d] = self.pool.alloc(n)
            elif kind == "dummy_free":
                _, d = op
                self.pool.free(self.dummies.pop(d))
            elif kind == "write":
                counts = np.asarray(op[1], dtype=np.int32)
                self.write_tokens(op_index, counts, values, stream)
            elif kind == "prompt":
                _, s, tokens = op
                self.admit_prompt(op_index, s, tokens, values, stream)
            else:
                raise ValueError(kind)
        self.upload_tables()

    def write_tokens(self, op_index: int, counts: np.ndarray, values: str = "numpy", stream=None):
        """Append counts[s] tokens to each sequence (a multi-token write through a3..a5)."""
        w = self.w
        total = int(counts.sum())
        slots, pairs = self.pool.prepare_append(self.tables, self.lens, counts)
        slots_d = torch.from_numpy(slots.copy()).to(self.device)
        if len(pairs):
            self.pool.copy_blocks(torch.from_numpy(pairs.copy()).to(self.device), status=self.status, stream=stream)
            self.cow_log.append(pairs.copy())
        for layer in range(w.num_layers):
            if values == "numpy":
                kn = torch.from_numpy(wl.write_values(w, op_index, layer, 0, total)).to(self.device)
                vn = torch.from_numpy(wl.write_values(w, op_index, layer, 1, total)).to(self.device)
            else:
                kn = wl.torch_normal_fp16(w.seed, (400, op_index, layer), (total, w.num_heads, w.head_dim), self.device)
                vn = wl.torch_normal_fp16(w.seed, (401, op_index, layer), (total, w.num_heads, w.head_dim), self.device)
            self.pool.append(layer, kn, vn, slots_d, status=self.status, stream=stream)
        self.last_pairs, self.last_slots = pairs.copy(), slots.copy()
        return slots, pairs

    def admit_prompt(self, op_index: int, s: int, tokens, values: str = "numpy", stream=None):
        """Sequence s arrives with prompt ``tokens``: cached leading blocks are shared
        (pkv_prefix_lookup), the remaining tokens are written through the append
        path, and the prompt's full blocks are registered (pkv_prefix_register)."""
        w, B = self.w, self.w.block_size
        hashes = bd.prompt_block_hashes(tokens, B)
        hit = self.pool.prefix_lookup(hashes)
        self.tables[s, :len(hit)] = hit
        self.lens[s] = len(hit) * B
        n_new = len(tokens) - len(hit) * B
        counts = np.zeros(w.num_seqs, dtype=np.int32)
        counts[s] = n_new
        self.write_tokens(op_index, counts, values, stream)
        full = len(hashes)
        if full > len(hit):
            self.pool.prefix_register(hashes[len(hit):], self.tables[s, len(hit):full])

    # ------------------------------------------------------------------ swap (preemption)
    def swap_out(self, s: int, host_buf, staging=None, stream=None) -> int:
        """Move sequence s's blocks (all layers) to ``host_buf`` (pinned uint8), then release
        them; its length is kept. With a device ``staging`` buffer the blocks are gathered there
        and copied to the host; without one the gather kernel writes ``host_buf`` directly over
        the host link. Returns the number of blocks."""
        w, B = self.w, self.w.block_size
        n = -(-int(self.lens[s]) // B)
        ids = self.tables[s, :n].copy()
        nbytes = n * self.pool.swap_bytes_per_block()
        st = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(st):
            blocks = torch.from_numpy(ids).to(self.device, non_blocking=False)
            if staging is None:
                self.pool.gather_blocks(blocks, host_buf, status=self.status, stream=st)
            else:
                self.pool.gather_blocks(blocks, staging, status=self.status, stream=st)
                host_buf[:nbytes].copy_(staging[:nbytes], non_blocking=True)
        self.pool.free(ids)
        self.tables[s, :] = -1
        return n

    def swap_in(self, s: int, n: int, host_buf, staging=None, stream=None) -> None:
        """Bring sequence s's n swapped blocks back into freshly allocated blocks (through the
        device ``staging`` buffer if one is given, else read from ``host_buf`` by the kernel)."""
        ids = self.pool.alloc(n)
        self.tables[s, :n] = ids
        nbytes = n * self.pool.swap_bytes_per_block()
        st = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(st):
            blocks = torch.tensor(ids, dtype=torch.int32, device=self.device)
            if staging is None:
                self.pool.scatter_blocks(blocks, host_buf, status=self.status, stream=st)
            else:
                staging[:nbytes].copy_(host_buf[:nbytes], non_blocking=True)
                self.pool.scatter_blocks(blocks, staging, status=self.status, stream=st)

    def upload_tables(self):
        self.tables_d.copy_(torch.from_numpy(self.tables))
        self.lens_d.copy_(torch.from_numpy(self.lens))
        if self.cascade:
            groups = np.zeros((max(self.w.num_seqs, 1), 4), dtype=np.int32)
            begin = np.zeros(max(self.w.num_seqs, 1), dtype=np.int32)
            self._plan(groups, begin)
            self.groups_d.copy_(torch.from_numpy(groups))
            self.begin_d.copy_(torch.from_numpy(begin))

    def _plan(self, groups_out: np.ndarray, begin_out: np.ndarray) -> None:
        """Cascade plan of the current host tables and lengths into the given buffers."""
        g, _ = bd.cascade_plan(self.tables, self.lens, self.w.block_size, groups_out=groups_out,
                               begin_out=begin_out[: self.w.num_seqs])
        self.plan_groups = len(g)
        self.plan = g.copy()
        self.plan_prefix = int(g[:, 2].max()) if len(g) else 0
        self.plan_splits = bd.prefix_splits(len(g), self.w.num_heads, self.plan_prefix) if len(g) else 0

    # ------------------------------------------------------------------ decode step
    def prepare_step(self, stream=None):
        """Host half of a decode step plus its H2D copies (enqueued on ``stream``)."""
        st = self._stage[self._buf]
        if st["event"] is not None:
            st["event"].synchronize()       # staging buffer no longer read by an older step
        slots, pairs = self.pool.prepare_append(self.tables, self.lens, None,
                                                slot_out=st["slots"].numpy(), pair_out=st["pairs"].numpy())
        st["tables"].numpy()[...] = self.tables
        st["lens"].numpy()[...] = self.lens
        if self.cascade:
            self._plan(st["groups"].numpy(), st["begin"].numpy())
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.tables_d.copy_(st["tables"], non_blocking=True)
            self.lens_d.copy_(st["lens"], non_blocking=True)
            if self.cascade:
                if self.plan_groups:
                    self.groups_d[: self.plan_groups].copy_(st["groups"][: self.plan_groups], non_blocking=True)
                self.begin_d.copy_(st["begin"], non_blocking=True)
            self.slots_d[: len(slots)].copy_(st["slots"][: len(slots)], non_blocking=True)
            if len(pairs):
                self.pairs_d[: len(pairs)].copy_(st["pairs"][: len(pairs)], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s)
        st["event"] = ev
        self._buf ^= 1
        self.last_pairs, self.last_slots = pairs.copy(), slots.copy()
        return len(slots), len(pairs)

    def device_step(self, q, k_new, v_new, out, n_slots: int, n_pairs: int, stream=None,
                    attn_events: Optional[list] = None, scale: float = 0.0):
        """Device half of a decode step: COW copies, then per layer append + attention.

        q, k_new, v_new, out: contiguous fp16 [L, S, H, D] on the device.
        ``attn_events`` (optional) gets (start, end) CUDA events around each
        layer's attention launch. Arguments are marshalled once per step; each
        launch is one C call.
        """
        w = self.w
        L = bd.lib()
        s = stream if stream is not None else torch.cuda.current_stream()
        sp = s.cuda_stream
        for t in (q, k_new, v_new, out):
            if t.dtype != torch.float16 or not t.is_contiguous() or t.shape[0] != w.num_layers:
                raise ValueError("step tensors must be contiguous fp16 [L, S, H, D]")
        h = self.pool.handle
        status = self.status.data_ptr()
        if n_pairs:
            bd.check(L.pkv_copy_blocks(h, self.pairs_d.data_ptr(), n_pairs, status, sp))
        row = w.num_seqs * w.num_heads * w.head_dim * 2
        qp, kp, vp, op = q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), out.data_ptr()
        tp, lp, slp = self.tables_d.data_ptr(), self.lens_d.data_ptr(), self.slots_d.data_ptr()
        wsp, wsb = self.workspace.data_ptr(), self.workspace.numel()
        maxb, S = w.max_blocks, w.num_seqs
        sc = float(scale)
        fused = self.fused and n_slots == S
        early = bd.ATTN_INPUTS_EARLY
        # after the layer's own append launch of one token per sequence (which first waits for
        # everything before it on the stream): the attention may start early, the tiles holding
        # the appended rows read last
        after_append = bd.ATTN_INPUTS_EARLY | bd.ATTN_LAST_ROW_PENDING if n_slots == S else 0
        G, splits = (self.plan_groups, self.plan_splits) if self.cascade else (0, 0)
        if G:
            gp, bp = self.groups_d.data_ptr(), self.begin_d.data_ptr()
            pp, pb = self.pieces.data_ptr(), self.pieces.numel()
        for layer in range(w.num_layers):
            off = layer * row
            if attn_events is not None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
            if G:
                # the shared prefixes once per group, then each sequence's private rest (+ append);
                # layers after the first follow the previous layer's private pass, which writes
                # none of the groups, tables or this layer's cache: the prefix pass starts early
                bd.check(L.pkv_prefix_attention(h, layer, qp + off, gp, G, splits, tp, maxb, S, sc, pp, pb, status,
                                                bd.ATTN_INPUTS_EARLY if layer > 0 else 0, sp))
                if not fused:
                    bd.check(L.pkv_append(h, layer, kp + off, vp + off, slp, n_slots, status, sp))
                # after the prefix pass (which writes only pieces) or the append, the private
                # pass may start early
                bd.check(L.pkv_decode_attention_ex(h, layer, qp + off, kp + off if fused else None,
                                                   vp + off if fused else None, slp if fused else None, tp, maxb,
                                                   lp, S, bp, pp, splits, sc, op + off, wsp, wsb,
                                                   bd.ATTN_INPUTS_EARLY if fused else after_append, sp))
            elif fused:
                # layers after the first follow the previous layer's attention, which writes
                # none of this layer's tables, lengths or cache: start early
                bd.check(L.pkv_decode_attention_ex(h, layer, qp + off, kp + off, vp + off, slp, tp, maxb, lp, S,
                                                   None, None, 0, sc, op + off, wsp, wsb,
                                                   early if layer > 0 else 0, sp))
            else:
                bd.check(L.pkv_append(h, layer, kp + off, vp + off, slp, n_slots, status, sp))
                bd.check(L.pkv_decode_attention_ex(h, layer, qp + off, None, None, None, tp, maxb, lp, S,
                                                   None, None, 0, sc, op + off, wsp, wsb, after_append, sp))
            if attn_events is not None:
                e1.record(s)
                attn_events.append((e0, e1))

    def capture(self, q, k_new, v_new, out, scale: float = 0.0):
        """Capture the device half of a decode step without COW copies into a CUDA graph.

        The graph holds, per layer, the append and the attention launches on the
        fixed device buffers (tables, lengths, slots, q, k_new, v_new, out);
        :meth:`step_graph` refreshes those buffers and replays it.
        """
        w = self.w
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            # first launches (attribute and occupancy queries) happen outside capture
            self.device_step(q, k_new, v_new, out, w.num_seqs, 0, side, scale=scale)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            self.device_step(q, k_new, v_new, out, w.num_seqs, 0, None, scale=scale)
        torch.cuda.synchronize()
        self._graph = g
        self._graph_tensors = (q, k_new, v_new, out)
        self._graph_scale = scale
        self._graph_plan = (self.plan_groups, self.plan_splits)
        return g

    def step_graph(self, stream=None):
        """A decode step replaying the captured graph (COW copies, if any, run first).

        The graph bakes in the cascade plan's shape (groups, splits); a step
        whose plan has another shape re-captures first.
        """
        n_slots, n_pairs = self.prepare_step(stream)
        if n_slots != self.w.num_seqs:
            raise RuntimeError("the captured step appends one token per sequence")
        if (self.plan_groups, self.plan_splits) != self._graph_plan:
            s = stream if stream is not None else torch.cuda.current_stream()
            s.synchronize()
            self.capture(*self._graph_tensors, scale=self._graph_scale)
        s = stream if stream is not None else torch.cuda.current_stream()
        if n_pairs:
            bd.check(bd.lib().pkv_copy_blocks(self.pool.handle, self.pairs_d.data_ptr(), n_pairs,
                                              self.status.data_ptr(), s.cuda_stream))
        with torch.cuda.stream(s):
            self._graph.replay()
        return n_slots, n_pairs

    def attention(self, layer: int, q, out, stream=None, scale: float = 0.0, early: bool = False):
        """One layer's decode attention over the current tables (q, out: fp16 [L, S, H, D]).

        ``early``: the preceding launch on the stream is an attention launch of this
        engine (it writes none of the tables, lengths or cache), so this one may
        start reading before it ends.
        """
        w = self.w
        s = stream if stream is not None else torch.cuda.current_stream()
        off = layer * w.num_seqs * w.num_heads * w.head_dim * 2
        if self.cascade and self.plan_groups:
            L, S = bd.lib(), w.num_seqs
            bd.check(L.pkv_prefix_attention(self.pool.handle, layer, q.data_ptr() + off, self.groups_d.data_ptr(),
                                            self.plan_groups, self.plan_splits, self.tables_d.data_ptr(),
                                            w.max_blocks, S, float(scale), self.pieces.data_ptr(),
                                            self.pieces.numel(), self.status.data_ptr(),
                                            bd.ATTN_INPUTS_EARLY if early else 0, s.cuda_stream))
            bd.check(L.pkv_decode_attention_ex(
                self.pool.handle, layer, q.data_ptr() + off, None, None, None, self.tables_d.data_ptr(),
                w.max_blocks, self.lens_d.data_ptr(), S, self.begin_d.data_ptr(), self.pieces.data_ptr(),
                self.plan_splits, float(scale), out.data_ptr() + off, self.workspace.data_ptr(),
                self.workspace.numel(), bd.ATTN_INPUTS_EARLY, s.cuda_stream))
            return
        if early:
            bd.check(bd.lib().pkv_decode_attention_ex(
                self.pool.handle, layer, q.data_ptr() + off, None, None, None, self.tables_d.data_ptr(),
                w.max_blocks, self.lens_d.data_ptr(), w.num_seqs, None, None, 0, float(scale), out.data_ptr() + off,
                self.workspace.data_ptr(), self.workspace.numel(), bd.ATTN_INPUTS_EARLY, s.cuda_stream))
            return
        bd.check(bd.lib().pkv_pool_decode_attention(
            self.pool.handle, layer, q.data_ptr() + off, self.tables_d.data_ptr(), w.max_blocks,
            self.lens_d.data_ptr(), w.num_seqs, float(scale), out.data_ptr() + off, self.workspace.data_ptr(),
            self.workspace.numel(), s.cuda_stream))

    def step(self, q, k_new, v_new, out, stream=None, attn_events=None, scale: float = 0.0):
        n_slots, n_pairs = self.prepare_step(stream)
        self.device_step(q, k_new, v_new, out, n_slots, n_pairs, stream, attn_events, scale)
        return n_slots, n_pairs

    # ------------------------------------------------------------------ inputs and checks
    def step_inputs(self, step: int, values: str = "numpy"):
        """q, k_new, v_new for every layer of ``step``: fp16 [L, S, H, D] on the device."""
        w = self.w
        if values == "numpy":
            q = np.stack([wl.query_values(w, step, l) for l in range(w.num_layers)])
            k = np.stack([wl.new_token_values(w, step, l, 0) for l in range(w.num_layers)])
            v = np.stack([wl.new_token_values(w, step, l, 1) for l in range(w.num_layers)])
            return tuple(torch.from_numpy(a).to(self.device) for a in (q, k, v))
        shp = (w.num_layers, w.num_seqs, w.num_heads, w.head_dim)
        return tuple(wl.torch_normal_fp16(w.seed, (tag, step), shp, self.device) for tag in (200, 300, 301))

    def device_status(self) -> int:
        a = int(self.status[0].item()) & 0xFFFFFFFF
        b = bd.workspace_status(self.workspace)
        return a | b

    def kv_bytes_per_layer(self) -> int:
        """Algorithmic K+V bytes one attention launch reads (current lengths)."""
        return int(self.lens.astype(np.int64).sum()) * self.w.kv_bytes_per_token_layer

    def unique_kv_bytes_per_layer(self) -> int:
        """K+V bytes of the distinct tokens a layer's attention covers: every sequence's
        context, minus all but one copy of each group's shared prefix (the cascade plan)."""
        dup = sum((int(n) - 1) * int(P) for _, n, P, _ in self.plan.tolist()) if self.cascade else 0
        return (int(self.lens.astype(np.int64).sum()) - dup) * self.w.kv_bytes_per_token_layer
