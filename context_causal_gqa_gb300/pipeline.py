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
    """

    def __init__(self, w, inputs, device="cuda", schedule="ring", fused=False):
        load()
        if schedule not in ("ring", "a2a"):
            raise ValueError(schedule)
        self.w = w
        self.x = inputs
        self.device = device
        self.schedule = schedule
        self.fused = fused or schedule == "a2a"
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
            self.lse = torch.empty((g, T, hq // g), dtype=torch.float32, device=device)
            self.dqs = torch.empty_like(self.qs)
            self.dks = torch.empty_like(self.ks)
            self.dvs = torch.empty_like(self.vs)
        else:
            self.os = torch.empty((T, hq, D), **e)
            self.lse = torch.empty((T, hq), dtype=torch.float32, device=device)
            self.dqs = torch.empty((T, hq, D), **e)
            self.dks = torch.empty((T, hkv, D), **e)
            self.dvs = torch.empty((T, hkv, D), **e)
        # outputs in the caller's layout
        self.o = torch.empty((T, hq, D), **e) if self.split else self.os
        self.dq = torch.empty((T, hq, D), **e) if self.split else self.dqs
        self.dk = torch.empty((T, hkv, D), **e) if self.split else self.dks
        self.dv = torch.empty((T, hkv, D), **e) if self.split else self.dvs
        self.launches_per_step = None

    def run(self, stream=None):
        """Enqueue one step; returns the number of kernels it launched."""
        x, w, n = self.x, self.w, 0
        cu, cpad = x["cu_seqlens"], x["cu_seqlens_padded"]
        kw = dict(status=self.status, stream=stream, check=False)
        if self.split:
            for src, dst in ((x["q"], self.qs), (x["k"], self.ks), (x["v"], self.vs), (x["do"], self.dos)):
                thd_pack(src, cpad, w.cp, out=dst, **kw)
                n += last_launch_count()
            q, k, v, do, hg = self.qs, self.ks, self.vs, self.dos, w.cp
        else:
            q, k, v, do, hg = x["q"], x["k"], x["v"], x["do"], 1
        attn_fwd(q, k, v, cu, cpad, self.attn_cp, head_groups=hg, out=self.os, lse=self.lse, workspace=self.ws_f,
                 fused=self.fused, **kw)
        n += last_launch_count()
        attn_bwd(q, k, v, self.os, do, self.lse, cu, cpad, self.attn_cp, head_groups=hg, dq=self.dqs, dk=self.dks,
                 dv=self.dvs, workspace=self.ws_b, **kw)
        n += last_launch_count()
        if self.split:
            for src, dst in ((self.os, self.o), (self.dqs, self.dq), (self.dks, self.dk), (self.dvs, self.dv)):
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
        return [self.x["q"], self.x["k"], self.x["v"], self.x["do"]]

    def output_tensors(self):
        return [self.o, self.lse, self.dq, self.dk, self.dv]

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
