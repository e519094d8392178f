"""One full pass of the CP-emulated attention path over a workload.

A step is: (for the A2A workload) pack q, k, v, dO from the rank-major local
layout into the head-split layout; forward (CP split + ring-step partials +
LSE merge); backward (Delta dot, dQ pass, dK/dV pass); (A2A) unpack o, dQ,
dK, dV back to the rank-major layout.  Every buffer, the workspaces and the
status word are allocated once, so that a step launches only this library's
kernels and never synchronises.
"""

import ctypes

import torch

from . import (Workspace, attn_bwd, attn_fwd, get_status, last_launch_count, load, thd_pack, thd_unpack,
               CCGError)


# Copies between pinned host memory and the device are split into this many
# contiguous pieces on as many streams, so that several copy engines share
# each direction.
COPY_LANES = 4


def _copy_lanes(dsts, srcs, lanes):
    """dst[i].copy_(src[i]) for every pair, each tensor cut into len(lanes)
    contiguous pieces copied on their own streams; lanes[0] waits for all."""
    lead = lanes[0]
    for s in lanes[1:]:
        s.wait_stream(lead)
    for d, h in zip(dsts, srcs):
        dv, hv = d.view(-1), h.view(-1)
        n = dv.numel()
        step = (n + len(lanes) - 1) // len(lanes)
        for i, s in enumerate(lanes):
            lo, hi = i * step, min(n, (i + 1) * step)
            if lo >= hi:
                continue
            with torch.cuda.stream(s):
                dv[lo:hi].copy_(hv[lo:hi], non_blocking=True)
    for s in lanes[1:]:
        lead.wait_stream(s)


class IOSet:
    """One set of the step's caller-facing device buffers: inputs x (dict of
    q, k, v, do) and outputs o, lse, dq, dk, dv."""

    def __init__(self, x, o, lse, dq, dk, dv):
        self.x, self.o, self.lse, self.dq, self.dk, self.dv = x, o, lse, dq, dk, dv

    def inputs(self):
        return [self.x["q"], self.x["k"], self.x["v"], self.x["do"]]

    def outputs(self):
        return [self.o, self.lse, self.dq, self.dk, self.dv]


class AttentionStep:
    """Preallocated forward + backward over one workload on one device.

    inputs: dict with q [T,Hq,D], k/v [T,Hkv,D], do [T,Hq,D] (bf16, on
    `device`), cu_seqlens and cu_seqlens_padded (int32).  With the A2A round
    trip (w.pack_roundtrip) the inputs are in the rank-major local layout and
    the outputs come back in it; otherwise everything is plain packed THD.

    schedule: "ring" (default) -- the CP-emulated ring over w.cp ranks on the
    (possibly head-split) layout; "a2a" -- the A2A (Ulysses-style) schedule:
    pack to w.cp head groups, full-sequence attention per head group (CP = 1,
    no partials, no merge), unpack.  fused: forward with one online softmax
    over all ring steps (ccg_attn_fwd_fused) instead of partials + merge.
    head_parts: P > 1 runs the ring forward and merge over P head parts in
    turn (a workspace sized for Hq/P heads).  keep_ds: give the backward the
    workload's longest padded sequence as its length bound, which at D = 256
    selects the backward that keeps dS for the dK pass.

    The caller-facing buffers (inputs, o, lse, dq, dk, dv) form an IOSet; a
    second set is allocated on demand for the host pipeline, in which the
    copies of one step overlap the compute of its neighbours.
    """

    def __init__(self, w, inputs, device="cuda", schedule="ring", fused=False, head_parts=0, keep_ds=False):
        load()
        if schedule not in ("ring", "a2a"):
            raise ValueError(schedule)
        self.w = w
        self.x = inputs
        self.device = device
        self.schedule = schedule
        self.fused = fused or schedule == "a2a"
        self.head_parts = head_parts
        self.max_seqlen = int(max(w.padded)) if keep_ds and w.padded else 0
        self.attn_cp = 1 if schedule == "a2a" else w.cp
        T, hq, hkv, D, cp = w.total_tokens, w.hq, w.hkv, w.head_dim, w.cp
        self.split = bool(w.pack_roundtrip) or schedule == "a2a"
        e = dict(dtype=torch.bfloat16, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws_f = Workspace(device)
        self.ws_b = Workspace(device)
        if self.split:
            g = cp
            self.qs = torch.empty((g, T, hq // g, D), **e)
            self.ks = torch.empty((g, T, hkv // g, D), **e)
            self.vs = torch.empty((g, T, hkv // g, D), **e)
            self.dos = torch.empty((g, T, hq // g, D), **e)
            self.os = torch.empty_like(self.qs)
            self.dqs = torch.empty_like(self.qs)
            self.dks = torch.empty_like(self.ks)
            self.dvs = torch.empty_like(self.vs)
        self.io = [self._new_io(inputs)]
        io = self.io[0]
        self.o, self.lse, self.dq, self.dk, self.dv = io.o, io.lse, io.dq, io.dk, io.dv
        self.launches_per_step = None
        self._pipe = None

    def _new_io(self, x=None):
        w, dev = self.w, self.device
        T, hq, hkv, D, g = w.total_tokens, w.hq, w.hkv, w.head_dim, w.cp
        e = dict(dtype=torch.bfloat16, device=dev)
        if x is None:
            x = dict(self.x)
            for name in ("q", "k", "v", "do"):
                x[name] = torch.empty_like(self.x[name])
        # LSE stays in the attention's grouping (head-split when split)
        lse = (torch.empty((g, T, hq // g), dtype=torch.float32, device=dev) if self.split
               else torch.empty((T, hq), dtype=torch.float32, device=dev))
        return IOSet(x, torch.empty((T, hq, D), **e), lse, torch.empty((T, hq, D), **e),
                     torch.empty((T, hkv, D), **e), torch.empty((T, hkv, D), **e))

    def run(self, stream=None, io=None):
        """Enqueue one step on `io` (default: the first set); returns the
        number of kernels it launched."""
        io = self.io[0] if io is None else io
        x, w, n = io.x, self.w, 0
        cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
        kw = dict(status=self.status, stream=stream, check=False)
        if self.split:
            for src, dst in ((x["q"], self.qs), (x["k"], self.ks), (x["v"], self.vs), (x["do"], self.dos)):
                thd_pack(src, cpad, w.cp, out=dst, **kw)
                n += last_launch_count()
            q, k, v, do, hg = self.qs, self.ks, self.vs, self.dos, w.cp
            o, dq, dk, dv = self.os, self.dqs, self.dks, self.dvs
        else:
            q, k, v, do, hg = x["q"], x["k"], x["v"], x["do"], 1
            o, dq, dk, dv = io.o, io.dq, io.dk, io.dv
        attn_fwd(q, k, v, cu, cpad, self.attn_cp, head_groups=hg, out=o, lse=io.lse, workspace=self.ws_f,
                 fused=self.fused, head_parts=self.head_parts, **kw)
        n += last_launch_count()
        attn_bwd(q, k, v, o, do, io.lse, cu, cpad, self.attn_cp, head_groups=hg, dq=dq, dk=dk, dv=dv,
                 workspace=self.ws_b, max_seqlen=self.max_seqlen, **kw)
        n += last_launch_count()
        if self.split:
            for src, dst in ((self.os, io.o), (self.dqs, io.dq), (self.dks, io.dk), (self.dvs, io.dv)):
                thd_unpack(src, cpad, w.cp, out=dst, **kw)
                n += last_launch_count()
        self.launches_per_step = n
        return n

    def check(self, stream=None):
        code = get_status(self.status, stream)
        if code != 0:
            raise CCGError(code, "AttentionStep (device status)")

    # ------------------------------------------------------------ host I/O
    def input_tensors(self):
        return self.io[0].inputs()

    def output_tensors(self):
        return self.io[0].outputs()

    def run_from_host(self, host_in, host_out, stream=None):
        """End-to-end step from pinned host buffers: H2D of q, k, v, dO, the
        step, then D2H of o, lse, dq, dk, dv (all on one stream)."""
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            for d, h in zip(self.input_tensors(), host_in):
                d.copy_(h, non_blocking=True)
            n = self.run(stream=s)
            for h, d in zip(host_out, self.output_tensors()):
                h.copy_(d, non_blocking=True)
        return n

    def run_from_host_pipelined(self, host_in, host_out, steps, stream=None):
        """`steps` end-to-end steps from pinned host buffers with the copies
        overlapped: step i computes on `stream` from IOSet i % 2 while the
        H2D of step i+1's inputs runs on the copy-in streams and the D2H of
        step i-1's outputs on the copy-out streams.  Every step copies its full inputs
        in and its full outputs out.  Returns (start, end) CUDA events that
        bracket all copies and compute; nothing is synchronised."""
        if len(self.io) < 2:
            self.io.append(self._new_io())
        if self._pipe is None:
            mk = lambda: [torch.cuda.Stream(self.device) for _ in range(COPY_LANES)]  # noqa: E731
            self._pipe = (mk(), mk())
        lanes_in, lanes_out = self._pipe
        s_in, s_out = lanes_in[0], lanes_out[0]
        s_c = torch.cuda.current_stream() if stream is None else stream
        ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
        h2d = [ev(), ev()]
        comp = [ev(), ev()]
        d2h = [ev(), ev()]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_c)
        s_in.wait_event(start)
        for i in range(steps):
            b = i % 2
            io = self.io[b]
            if i >= 2:
                s_in.wait_event(comp[b])           # step i-2 has finished with these inputs
            _copy_lanes(io.inputs(), host_in, lanes_in)
            h2d[b].record(s_in)
            s_c.wait_event(h2d[b])
            if i >= 2:
                s_c.wait_event(d2h[b])             # step i-2's outputs have been copied out
            self.run(stream=s_c, io=io)
            comp[b].record(s_c)
            s_out.wait_event(comp[b])
            _copy_lanes(host_out, io.outputs(), lanes_out)
            d2h[b].record(s_out)
        s_c.wait_event(d2h[(steps - 1) % 2])
        if steps >= 2:
            s_c.wait_event(d2h[(steps - 2) % 2])
        end.record(s_c)
        return start, end

    def host_buffers(self):
        ins = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in self.input_tensors()]
        outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in self.output_tensors()]
        return ins, outs

    def io_bytes(self):
        bi = sum(t.numel() * t.element_size() for t in self.input_tensors())
        bo = sum(t.numel() * t.element_size() for t in self.output_tensors())
        return bi, bo


def profile_begin(capacity):
    code = load().ccg_profile_begin(int(capacity))
    if code != 0:
        raise CCGError(code, "ccg_profile_begin")


def profile_end():
    """Stop recording and return [(kernel name, ms)] for every timed launch."""
    lib = load()
    lib.ccg_profile_end()
    out = []
    name = ctypes.c_char_p()
    ms = ctypes.c_float()
    for i in range(lib.ccg_profile_count()):
        code = lib.ccg_profile_get(i, ctypes.byref(name), ctypes.byref(ms))
        if code != 0:
            raise CCGError(code, "ccg_profile_get")
        out.append((name.value.decode(), float(ms.value)))
    return out
