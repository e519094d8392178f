"""GB300-native context-parallel causal GQA attention over packed THD BF16.

Thin Python binding over the C ABI of libccg (include/ccg.h).  PyTorch is
used for device memory and streams only: every step of the path runs in the
library's CUDA kernels, and every call raises if the library is missing or
returns an error.  There is no CPU or PyTorch fallback.
"""

import ctypes
import math

from ._lib import AttnDesc, load

__all__ = ["AttnDesc", "CCGError", "load", "make_desc", "workspace_size", "attn_fwd", "attn_fwd_step",
           "attn_bwd", "cp_split", "cp_lse_merge", "bwd_dot", "thd_pack", "thd_unpack", "get_status",
           "status_str", "last_launch_count", "Workspace"]

STATUS = {0: "CCG_OK", 1: "CCG_ERR_INVALID_ARG", 2: "CCG_ERR_UNSUPPORTED", 3: "CCG_ERR_ALIGNMENT",
          4: "CCG_ERR_WORKSPACE", 5: "CCG_ERR_SEQLENS", 6: "CCG_ERR_TIMEOUT", 7: "CCG_ERR_CUDA"}


class CCGError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_str(code)})")


def _check(code, where):
    if code != 0:
        raise CCGError(code, where)


def status_str(code):
    return load().ccg_status_str(int(code)).decode()


def last_launch_count():
    return int(load().ccg_last_launch_count())


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_desc(batch, hq, hkv, head_dim, cp, total_tokens, head_groups=1, scale=0.0, pitches=(0, 0, 0, 0),
              head_parts=0, max_seqlen=0):
    """pitches: row pitch in elements of q, k, v, dO (0 = dense); head_parts:
    P > 1 runs the ring forward and merge over P head parts in turn;
    max_seqlen > 0 (a bound on every padded sequence length) selects the
    D = 256 backward that keeps dS for the dK pass."""
    return AttnDesc(batch=batch, hq=hq, hkv=hkv, head_dim=head_dim, causal=1, cp=cp,
                    head_groups=head_groups, head_parts=head_parts, total_tokens=total_tokens, softmax_scale=scale,
                    q_pitch=pitches[0], k_pitch=pitches[1], v_pitch=pitches[2], do_pitch=pitches[3],
                    max_seqlen=max_seqlen)


def workspace_size(desc, kind):
    """kind: 0 / False forward, 1 / True backward, 2 fused forward."""
    return int(load().ccg_workspace_size(ctypes.byref(desc), int(kind)))


class Workspace:
    """Caller-owned device workspace (torch memory), grown on demand."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None

    def get(self, nbytes):
        import torch
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256) + 256, dtype=torch.uint8, device=self.device)
        base = self.buf.data_ptr()
        off = (-base) % 256
        return ctypes.c_void_p(base + off), self.buf.numel() - off


def _new_status(device):
    import torch
    return torch.zeros(1, dtype=torch.int32, device=device)


def _dense(t, name):
    """Outputs, o and lse are dense: a strided view there would be misread."""
    if t is not None and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _pitch(t, name):
    """Row pitch of a [T, H, D] input: 0 when dense, else its token stride
    (heads must stay contiguous, stride D; D contiguous)."""
    if t is None or t.dim() != 3:
        return 0
    T, H, D = t.shape
    if t.stride(2) != 1 or t.stride(1) != D:
        raise ValueError(f"{name}: heads and head_dim must be contiguous (strides (*, {D}, 1)), got {t.stride()}")
    return 0 if t.stride(0) == H * D or T <= 1 else t.stride(0)


def _desc_for(q, k, cu_seqlens, cp, head_groups, scale, v=None, do=None, head_parts=0, max_seqlen=0):
    hg = head_groups
    if q.dim() == 4:        # head-split [G][T][H/G][D]
        for t, name in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
            _dense(t, name)
        hg = q.shape[0]
        T, hq, D = q.shape[1], q.shape[0] * q.shape[2], q.shape[3]
        hkv = k.shape[0] * k.shape[2]
        pitches = (0, 0, 0, 0)
    else:
        T, hq, D = q.shape
        hkv = k.shape[1]
        pitches = (_pitch(q, "q"), _pitch(k, "k"), _pitch(v, "v"), _pitch(do, "do"))
    return make_desc(cu_seqlens.numel() - 1, hq, hkv, D, cp, T, hg, scale, pitches, head_parts, max_seqlen)


def attn_fwd(q, k, v, cu_seqlens, cu_seqlens_padded, cp, *, head_groups=1, scale=0.0, out=None, lse=None,
             workspace=None, status=None, stream=None, check=True, fused=False, head_parts=0):
    """Forward: returns (o, lse).  q [T,Hq,D] (or [G,T,Hq/G,D]), k/v likewise, bf16 on cuda.
    q, k, v may be row-strided views (e.g. slices of a fused QKV buffer); o is dense.
    fused=True runs ccg_attn_fwd_fused (one online softmax over all ring steps).
    head_parts=P > 1 runs the ring forward and merge over P head parts in turn
    with a workspace sized for Hq/P heads (bitwise the same result)."""
    import torch
    desc = _desc_for(q, k, cu_seqlens, cp, head_groups, scale, v=v, head_parts=head_parts)
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device) if out is None else _dense(out, "out")
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    _dense(lse, "lse")
    ws = workspace or Workspace(q.device)
    wptr, wbytes = ws.get(workspace_size(desc, 2 if fused else 0))
    st = _new_status(q.device) if status is None else status
    fn = load().ccg_attn_fwd_fused if fused else load().ccg_attn_fwd
    _check(fn(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(cu_seqlens_padded), _ptr(o),
              _ptr(lse), wptr, wbytes, _ptr(st), _stream(stream)), "ccg_attn_fwd_fused" if fused else "ccg_attn_fwd")
    if check:
        _check(get_status(st, stream), "ccg_attn_fwd (device)")
    return o, lse


def attn_fwd_step(q, k, v, cu_seqlens, cu_seqlens_padded, cp, step, o_part, lse_part, *, head_groups=1,
                  scale=0.0, workspace=None, status=None, stream=None, check=True):
    """One ring step's partial (o_part, lse_part), written in place (absent rows untouched)."""
    desc = _desc_for(q, k, cu_seqlens, cp, head_groups, scale, v=v)
    ws = workspace or Workspace(q.device)
    wptr, wbytes = ws.get(workspace_size(desc, False))
    st = _new_status(q.device) if status is None else status
    _check(load().ccg_attn_fwd_step(ctypes.byref(desc), step, _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens),
                                    _ptr(cu_seqlens_padded), _ptr(o_part), _ptr(lse_part), wptr, wbytes,
                                    _ptr(st), _stream(stream)), "ccg_attn_fwd_step")
    if check:
        _check(get_status(st, stream), "ccg_attn_fwd_step (device)")
    return o_part, lse_part


def attn_bwd(q, k, v, o, do, lse, cu_seqlens, cu_seqlens_padded, cp, *, head_groups=1, scale=0.0,
             dq=None, dk=None, dv=None, workspace=None, status=None, stream=None, check=True, max_seqlen=0):
    """Backward: returns (dq, dk, dv).  q, k, v, do may be row-strided views; o and the
    gradients are dense.  max_seqlen > 0: a bound on every padded sequence length,
    which selects the backward that keeps dS, and at D = 256 P (a larger workspace)."""
    import torch
    desc = _desc_for(q, k, cu_seqlens, cp, head_groups, scale, v=v, do=do, max_seqlen=max_seqlen)
    dense = lambda t: torch.empty(t.shape, dtype=t.dtype, device=t.device)  # noqa: E731
    dq = dense(q) if dq is None else _dense(dq, "dq")
    dk = dense(k) if dk is None else _dense(dk, "dk")
    dv = dense(v) if dv is None else _dense(dv, "dv")
    _dense(o, "o")
    _dense(lse, "lse")
    ws = workspace or Workspace(q.device)
    wptr, wbytes = ws.get(workspace_size(desc, True))
    st = _new_status(q.device) if status is None else status
    _check(load().ccg_attn_bwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                               _ptr(cu_seqlens), _ptr(cu_seqlens_padded), _ptr(dq), _ptr(dk), _ptr(dv),
                               wptr, wbytes, _ptr(st), _stream(stream)), "ccg_attn_bwd")
    if check:
        _check(get_status(st, stream), "ccg_attn_bwd (device)")
    return dq, dk, dv


def cp_split(cu_seqlens, cu_seqlens_padded, cp, total_tokens, *, status=None, stream=None, check=True):
    """Chunk table int32 [B][2cp][2] = (first physical row, length)."""
    import torch
    B = cu_seqlens.numel() - 1
    table = torch.empty((B, 2 * cp, 2), dtype=torch.int32, device=cu_seqlens.device)
    st = _new_status(cu_seqlens.device) if status is None else status
    _check(load().ccg_cp_split(_ptr(cu_seqlens), _ptr(cu_seqlens_padded), B, total_tokens, cp, _ptr(table),
                               _ptr(st), _stream(stream)), "ccg_cp_split")
    if check:
        _check(get_status(st, stream), "ccg_cp_split (device)")
    return table


def cp_lse_merge(o_parts, lse_parts, *, out=None, lse=None, stream=None):
    """K-way merge of partials o_parts[s] [..., D] bf16 with lse_parts[s] [...] float."""
    import torch
    K = len(o_parts)
    D = o_parts[0].shape[-1]
    rows = lse_parts[0].numel()
    o = torch.empty_like(o_parts[0]) if out is None else out
    lse = torch.empty_like(lse_parts[0]) if lse is None else lse
    op = (ctypes.c_void_p * K)(*[t.data_ptr() for t in o_parts])
    lp = (ctypes.c_void_p * K)(*[t.data_ptr() for t in lse_parts])
    _check(load().ccg_cp_lse_merge(K, op, lp, rows, D, _ptr(o), _ptr(lse), _stream(stream)), "ccg_cp_lse_merge")
    return o, lse


def bwd_dot(o, do, *, out=None, stream=None):
    import torch
    D = o.shape[-1]
    rows = o.numel() // D
    delta = torch.empty(o.shape[:-1], dtype=torch.float32, device=o.device) if out is None else out
    _check(load().ccg_bwd_dot(_ptr(o), _ptr(do), rows, D, _ptr(delta), _stream(stream)), "ccg_bwd_dot")
    return delta


def thd_pack(x, cu_seqlens_padded, cp, *, out=None, status=None, stream=None, check=True):
    """Rank-major [T,H,D] -> head-split [cp,T,H/cp,D]."""
    import torch
    T, H, D = x.shape
    out = torch.empty((cp, T, H // cp, D), dtype=x.dtype, device=x.device) if out is None else out
    st = _new_status(x.device) if status is None else status
    _check(load().ccg_thd_pack(_ptr(x), _ptr(cu_seqlens_padded), cu_seqlens_padded.numel() - 1, T, H, D, cp,
                               _ptr(out), _ptr(st), _stream(stream)), "ccg_thd_pack")
    if check:
        _check(get_status(st, stream), "ccg_thd_pack (device)")
    return out


def thd_unpack(x, cu_seqlens_padded, cp, *, out=None, status=None, stream=None, check=True):
    """Head-split [cp,T,H/cp,D] -> rank-major [T,H,D]."""
    import torch
    G, T, hg, D = x.shape
    out = torch.empty((T, G * hg, D), dtype=x.dtype, device=x.device) if out is None else out
    st = _new_status(x.device) if status is None else status
    _check(load().ccg_thd_unpack(_ptr(x), _ptr(cu_seqlens_padded), cu_seqlens_padded.numel() - 1, T, G * hg,
                                 D, cp, _ptr(out), _ptr(st), _stream(stream)), "ccg_thd_unpack")
    if check:
        _check(get_status(st, stream), "ccg_thd_unpack (device)")
    return out


def get_status(status, stream=None):
    return int(load().ccg_get_status(_ptr(status), _stream(stream)))
