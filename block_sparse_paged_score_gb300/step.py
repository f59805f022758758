"""One decode step of the sparse path as a single library call.

DecodeStep owns the step's caller-side buffers (row lengths, score rows,
selections, output, split-K workspace, error word) for a fixed batch shape and
runs ``bsp_sparse_decode_step`` -- write the new tokens, cast the queries to
e4m3 where the workload attends or scores in e4m3, row lengths, index
scores, top-k with the emitted sparse table, split-K attention and merge --
on one stream, without host synchronisation.

``HostDecodeStep`` is the end-to-end form a serving loop uses: the step's
inputs arrive in pinned host memory and its attention output must land
there.  Each direction either crosses by one copy-engine copy or is read or
written in place by the step's kernels (zero-copy).  ``MixedStep`` is the
chunked-prefill batch (decode rows first, then prefill chunks and pad rows)
as separate calls on one stream.
"""
import ctypes as C

import torch

from . import bsp


class DecodeStep:
    """select_in_scorer: hand the step a zeroed counter per (sequence, index
    head) so that the scorer's last CTA of each sequence selects its rows
    (where the library supports it; the outputs are the same, the step is
    slower on the benchmark workloads, so it is off by default)."""

    def __init__(self, w, kv, idx, block_table, device="cuda", flags=bsp.FORCE_TAIL, select_in_scorer=False):
        self.w = w
        self.kv, self.idx = kv, idx
        self.block_table = block_table
        tokens, rows = w.num_decode_tokens, w.num_decode_tokens * w.hkv
        self.tokens, self.rows = tokens, rows
        e = lambda *s, dt=torch.int32: torch.empty(s, dtype=dt, device=device)  # noqa: E731
        self.row_seq, self.row_len = e(rows), e(rows)
        self.scores = e(rows, w.max_pages, dt=torch.float32)
        self.topk_idx, self.sparse_bt, self.sparse_ctx = e(rows, w.k_pages), e(rows, w.k_pages), e(rows)
        self.out = e(tokens, w.hq, 128, dt=torch.bfloat16)
        self.q_cast = e(tokens, w.hq, 128, dt=torch.uint8)
        self.idx_q_cast = e(tokens, w.hidx, 128, dt=torch.uint8)
        self.ws = bsp.decode_workspace(rows, w.k_pages, w.group, device)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)
        self.args = bsp.DecodeStepArgs()
        a = self.args
        a.kv = C.pointer(kv.desc)
        a.idx = C.pointer(idx.desc)
        a.q_dtype, a.idx_q_dtype = w.q_dtype, w.idx_q_dtype
        a.q_cast, a.idx_q_cast = self.q_cast.data_ptr(), self.idx_q_cast.data_ptr()
        a.num_q_heads = w.hq
        a.num_seqs, a.q_len = w.num_decode, w.q_len
        a.block_table, a.bt_stride = block_table.data_ptr(), block_table.shape[1]
        a.max_pages, a.k_pages, a.flags, a.sm_scale = w.max_pages, w.k_pages, flags, w.sm_scale
        a.row_seq, a.row_len, a.scores = self.row_seq.data_ptr(), self.row_len.data_ptr(), self.scores.data_ptr()
        a.topk_idx, a.sparse_bt, a.sparse_ctx = (self.topk_idx.data_ptr(), self.sparse_bt.data_ptr(),
                                                 self.sparse_ctx.data_ptr())
        a.out, a.ws, a.ws_bytes, a.dev_err = self.out.data_ptr(), self.ws.data_ptr(), self.ws.numel(), \
            self.dev_err.data_ptr()
        self.sel_counters = torch.zeros(max(1, w.num_decode * w.hidx), dtype=torch.int32, device=device)
        a.sel_counters = self.sel_counters.data_ptr() if select_in_scorer else None

    def run(self, k_new, v_new, idx_k_new, slot, q, idx_q, seq_lens, events=None, stream=None):
        """Device tensors in; fills self.out (and the intermediate buffers)."""
        a = self.args
        a.k_new, a.v_new, a.idx_k_new, a.slot = (k_new.data_ptr(), v_new.data_ptr(), idx_k_new.data_ptr(),
                                                 slot.data_ptr())
        a.num_new_tokens = slot.numel()
        a.q, a.idx_q, a.seq_lens = q.data_ptr(), idx_q.data_ptr(), seq_lens.data_ptr()
        bsp.sparse_decode_step(a, events=events, stream=stream)
        return self.out


class HostDecodeStep:
    """End-to-end step: pinned host inputs -> device -> step -> host output.

    The step's inputs sit back to back (256-byte aligned) in one pinned host
    buffer.  `inputs` and `output` each choose how the bytes cross the link:
      "copy": one copy-engine copy (host-to-device of all the inputs, or
              device-to-host of the attention output) on the step's stream;
      "zero": no copy -- the step's kernels load the inputs straight from the
              pinned buffer, or the attention stores its output straight
              into pinned host memory (pinned memory is mapped into the
              device's address space; on a Grace-Blackwell node these loads
              and stores cross NVLink-C2C).
    zero_copy=True is inputs="zero", output="zero".  Works for a DecodeStep
    and for a MixedStep."""

    def __init__(self, step, host_inputs, device="cuda", zero_copy=False, inputs=None, output=None):
        self.step = step
        self.inputs = inputs or ("zero" if zero_copy else "copy")
        self.output = output or ("zero" if zero_copy else "copy")
        if "zero" in (self.inputs, self.output) and not isinstance(step, (DecodeStep, MixedStep)):
            raise ValueError("zero-copy transfer needs a DecodeStep or a MixedStep")
        offs, total = {}, 0
        for k, v in host_inputs.items():
            offs[k] = total
            total += (v.numel() * v.element_size() + 255) // 256 * 256
        self.nbytes = total
        self.host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dev_buf = torch.empty(total, dtype=torch.uint8, device=device)
        self.dev, self.host = {}, {}
        for k, v in host_inputs.items():
            n = v.numel() * v.element_size()
            self.host_buf[offs[k]:offs[k] + n].copy_(v.contiguous().view(-1).view(torch.uint8))
            self.dev[k] = self.dev_buf[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
            self.host[k] = self.host_buf[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
        self.out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()

    @property
    def h2d_bytes(self):
        return self.nbytes

    @property
    def d2h_bytes(self):
        return self.out_host.numel() * self.out_host.element_size()

    def run(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            if self.inputs == "copy":
                self.dev_buf.copy_(self.host_buf, non_blocking=True)
            d = self.dev if self.inputs == "copy" else self.host
            if self.output == "zero" and isinstance(self.step, MixedStep):
                # the step's attention launches store into the pinned output
                dev_out = self.step.out
                self.step.out = self.out_host
                try:
                    self.step.run(d["k"], d["v"], d["idx_k"], d["slot"], d["q"], d["idx_q"], d["seq_lens"], stream=s)
                finally:
                    self.step.out = dev_out
            elif self.output == "zero":
                a = self.step.args
                dev_out = a.out
                a.out = self.out_host.data_ptr()
                try:
                    self.step.run(d["k"], d["v"], d["idx_k"], d["slot"], d["q"], d["idx_q"], d["seq_lens"], stream=s)
                finally:
                    a.out = dev_out
            else:
                self.step.run(d["k"], d["v"], d["idx_k"], d["slot"], d["q"], d["idx_q"], d["seq_lens"], stream=s)
                self.out_host.copy_(self.step.out, non_blocking=True)
        return self.out_host


class MixedStep:
    """A chunked-prefill batch: decode rows first, then prefill chunks and pad
    rows (the vLLM forward's decode-first order).  Decode rows score on the
    mma.sync scorer and attend with split-K; prefill rows score on the tcgen05
    scorer and attend plan-free.  Same run() signature as DecodeStep; `events`
    (5 torch events) mark the same phases."""

    def __init__(self, w, kv, idx, block_table, device="cuda", flags=bsp.FORCE_TAIL):
        self.w, self.kv, self.idx, self.block_table = w, kv, idx, block_table
        self.flags = flags
        T, rows = w.num_tokens, w.num_rows
        self.nd_tok, self.nd = w.num_decode_tokens, w.num_decode_rows
        e = lambda *s, dt=torch.int32: torch.empty(s, dtype=dt, device=device)  # noqa: E731
        self.scores = e(rows, w.max_pages, dt=torch.float32)
        self.topk_idx, self.sparse_bt, self.sparse_ctx = e(rows, w.k_pages), e(rows, w.k_pages), e(rows)
        self.out = e(T, w.hq, 128, dt=torch.bfloat16)
        self.q_cast = e(T, w.hq, 128, dt=torch.uint8)
        self.idx_q_cast = e(T, w.hidx, 128, dt=torch.uint8)
        self.row_seq, self.row_len = e(rows), e(rows)
        self.ws = bsp.decode_workspace(max(self.nd, 1), w.k_pages, w.group, device)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)
        self.query_req_id = torch.from_numpy(w.query_req_id).to(device)
        self.query_abs_pos = torch.from_numpy(w.query_abs_pos).to(device)
        self.cu = torch.from_numpy(w.cu_prefill).to(device)
        self.num_chunks = len(w.cu_prefill) - 1
        self.max_tiles = bsp.prefill_tiles(w.cu_prefill)

    def run(self, k_new, v_new, idx_k_new, slot, q, idx_q, seq_lens, events=None, stream=None):
        w, nd, ndt = self.w, self.nd, self.nd_tok
        s = stream if stream is not None else torch.cuda.current_stream()
        mark = (lambda i: events[i].record(s)) if events is not None else (lambda i: None)  # noqa: E731
        mark(0)
        bsp.kv_page_write(self.kv, self.idx, k_new, v_new, idx_k_new, slot, self.dev_err, s)
        if w.q_dtype == bsp.FP8_E4M3:
            q = bsp.cast_e4m3(q, self.q_cast, s)
        if w.idx_q_dtype == bsp.FP8_E4M3:
            idx_q = bsp.cast_e4m3(idx_q, self.idx_q_cast, s)
        bsp.row_lengths_decode(seq_lens, w.q_len, w.hkv, self.row_seq[:nd], self.row_len[:nd], s)
        bsp.row_lengths_prefill(self.query_req_id, self.query_abs_pos, w.hkv, self.row_seq[nd:], self.row_len[nd:], s)
        mark(1)
        if nd:
            bsp.index_score(self.idx, idx_q[:ndt], w.idx_q_dtype, self.block_table, self.row_seq[:nd],
                            self.row_len[:nd], w.q_len, w.max_pages, self.scores[:nd], self.dev_err, s)
        bsp.index_score_prefill(self.idx, idx_q[ndt:], w.idx_q_dtype, self.block_table, self.row_seq[nd:],
                                self.row_len[nd:], self.cu, self.num_chunks, self.max_tiles, w.max_pages,
                                self.scores[nd:], self.dev_err, s)
        mark(2)
        bsp.topk_select(self.scores, self.row_seq, self.row_len, self.block_table, w.kv_dtype, w.k_pages,
                        self.flags, self.topk_idx, self.sparse_bt, self.sparse_ctx, s)
        mark(3)
        if nd:
            bsp.sparse_pa_decode(self.kv, q[:ndt], w.q_dtype, w.hq, self.sparse_bt[:nd], self.sparse_ctx[:nd],
                                 w.k_pages, w.sm_scale, self.out[:ndt], self.ws, self.dev_err, s)
        bsp.sparse_pa_prefill(self.kv, q[ndt:], w.q_dtype, w.hq, self.sparse_bt[nd:], self.sparse_ctx[nd:],
                              w.k_pages, w.sm_scale, self.out[ndt:], self.dev_err, s)
        mark(4)
        return self.out
