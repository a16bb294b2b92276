"""Python binding of the C ABI, with the same names.

Tensors are PyTorch CUDA tensors (device memory and streams only); each call
hands raw pointers and the current stream to libattnmask.  The binding does
no arithmetic of the method.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _native

ATTN_OK = 0
(ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE_TOO_SMALL, ATTN_ERR_MASK_MISMATCH,
 ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_DEVICE_INVALID_INPUT) = range(1, 8)
STATUS = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_WORKSPACE_TOO_SMALL", 4: "ATTN_ERR_MASK_MISMATCH", 5: "ATTN_ERR_CUDA",
    6: "ATTN_ERR_DEVICE_TIMEOUT", 7: "ATTN_ERR_DEVICE_INVALID_INPUT",
}
MASK_KINDS = {"causal": 0, "causal_document": 1, "shared_prefix": 2, "strip_thinking": 3,
              "strip_thinking_dup": 4, "none": 5, "dense": 6}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}
TILE_EMPTY, TILE_PARTIAL, TILE_FULL = 0, 1, 2
BLOCK_M = BLOCK_N = 128


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)} ({attn_status_string(status)})"
        if status == 5:
            msg += f": {attn_last_error_message()}"
        super().__init__(msg)


def _check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name: str, where: str, dtypes=None, shape=None, device=None) -> None:
    """Refuse, before any library call, a tensor the C side would misread: not
    on a CUDA device (a host pointer would reach a kernel), on another device
    than the rest, not contiguous (the layouts are dense row-major), of the
    wrong element type or shape."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise AttnError(1, f"{where}: {name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise AttnError(1, f"{where}: {name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise AttnError(1, f"{where}: {name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise AttnError(1, f"{where}: {name} has dtype {t.dtype}, expected one of {dtypes}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise AttnError(1, f"{where}: {name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _need_meta(where, cu_seqlens, seg_id, role, turn, dense_bits, dense_offsets, device=None):
    """cu_seqlens int32; seg_id / turn int32, role int8 (one value per token);
    the dense kind's words (32-bit) and int64 offsets."""
    _need(cu_seqlens, "cu_seqlens", where, (torch.int32,), device=device)
    dev = cu_seqlens.device
    _need(seg_id, "seg_id", where, (torch.int32,), device=dev)
    _need(role, "role", where, (torch.int8, torch.uint8), device=dev)
    _need(turn, "turn", where, (torch.int32,), device=dev)
    _need(dense_bits, "dense_bits", where, _WORD_DTYPES, device=dev)
    _need(dense_offsets, "dense_offsets", where, (torch.int64,), device=dev)


_WORD_DTYPES = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _kind(kind) -> int:
    return MASK_KINDS[kind] if isinstance(kind, str) else int(kind)


def attn_status_string(status: int) -> str:
    return _native.lib().attn_status_string(int(status)).decode()


def attn_last_error_message() -> str:
    return _native.lib().attn_last_error_message().decode()


def attn_version() -> int:
    return int(_native.lib().attn_version())


def attn_block_mask_workspace_size(batch: int, total_tokens: int, max_seqlen: int,
                                   block_m: int = BLOCK_M, block_n: int = BLOCK_N) -> int:
    out = ctypes.c_size_t(0)
    _check(_native.lib().attn_block_mask_workspace_size(batch, total_tokens, max_seqlen, block_m,
                                                        block_n, ctypes.byref(out)),
           "attn_block_mask_workspace_size")
    return int(out.value)


class BlockMask:
    """A built block mask: the C struct plus the tensors it points into."""

    # arrays attn_block_mask_build_noalloc keeps in its own scratch and does not
    # write to the workspace
    NOALLOC_UNWRITTEN = ("labels", "qt_off", "pair_off")

    def __init__(self, struct: _native.AttnBlockMask, workspace: torch.Tensor, keep: tuple,
                 noalloc: bool = False):
        self.struct = struct
        self.workspace = workspace
        self._keep = keep  # metadata tensors must outlive the mask
        self.noalloc = noalloc

    # -- read-back helpers (copy device arrays to the host; synchronising) --
    def _array(self, off: int, count: int, dtype) -> torch.Tensor:
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        raw = self.workspace[off: off + nbytes]
        return raw.view(dtype).cpu()

    def header(self) -> torch.Tensor:
        return self._array(self.struct.off_header, 16, torch.int32)

    @property
    def n_qtiles(self) -> int:
        return int(self.header()[0])

    def lists(self) -> dict:
        """Device arrays copied back: q-tile descriptors, labels, CSR lists, order.
        A mask from the no-allocation builder has no ``labels``, ``qt_off`` or
        ``pair_off`` (never written to its workspace); they are left out."""
        s = self.struct
        n = self.n_qtiles
        hdr = self.header()
        nent = int(hdr[1])
        koff = self._array(s.off_koff, n + 1, torch.int32)
        out = {
            "header": hdr,
            "qt_seq": self._array(s.off_qt_seq, n, torch.int32),
            "qt_idx": self._array(s.off_qt_idx, n, torch.int32),
            "labels": self._array(s.off_labels, s.max_qtiles * s.max_ktiles, torch.uint8)
                          .view(s.max_qtiles, s.max_ktiles)[:n],
            "kcount": self._array(s.off_kcount, n, torch.int32),
            "koff": koff,
            "kidx": self._array(s.off_kidx, nent, torch.int32),
            "klabel": self._array(s.off_klabel, nent, torch.uint8),
            "order": self._array(s.off_order, n, torch.int32),
            "qt_off": self._array(s.off_qt_off, s.batch + 1, torch.int32),
            "pair_off": self._array(s.off_pair_off, s.batch + 1, torch.int32),
            "pair_q0": self._array(s.off_pair_q0, int(hdr[3]), torch.int32),
            "pair_order": self._array(s.off_pair_order, int(hdr[3]), torch.int32),
            "qcount": self._array(s.off_qcount, n, torch.int32),
            "qoff": self._array(s.off_qoff, n + 1, torch.int32),
            "qidx": self._array(s.off_qidx, nent, torch.int32),
            "qlabel": self._array(s.off_qlabel, nent, torch.uint8),
            "korder": self._array(s.off_korder, n, torch.int32),
        }
        if self.noalloc:
            for name in self.NOALLOC_UNWRITTEN:
                del out[name]
        return out


def _params(role_think: int, dense_bits, dense_offsets) -> "_native.AttnMaskParams":
    return _native.AttnMaskParams(role_think, _ptr(dense_bits), _ptr(dense_offsets))


def attn_block_mask_build(kind, cu_seqlens: torch.Tensor, total_tokens: int, max_seqlen: int,
                          seg_id: Optional[torch.Tensor] = None, role: Optional[torch.Tensor] = None,
                          turn: Optional[torch.Tensor] = None, role_think: int = 1,
                          workspace: Optional[torch.Tensor] = None, stream=None,
                          dense_bits: Optional[torch.Tensor] = None,
                          dense_offsets: Optional[torch.Tensor] = None) -> BlockMask:
    """Build the block mask on the device (asynchronous on ``stream``)."""
    _need_meta("attn_block_mask_build", cu_seqlens, seg_id, role, turn, dense_bits, dense_offsets)
    _need(workspace, "workspace", "attn_block_mask_build", device=cu_seqlens.device)
    batch = cu_seqlens.numel() - 1
    need = attn_block_mask_workspace_size(batch, total_tokens, max_seqlen)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=cu_seqlens.device)
    params = _params(role_think, dense_bits, dense_offsets)
    out = _native.AttnBlockMask()
    _check(_native.lib().attn_block_mask_build(
        _kind(kind), ctypes.byref(params), _ptr(cu_seqlens), batch, total_tokens, max_seqlen,
        _ptr(seg_id), _ptr(role), _ptr(turn), BLOCK_M, BLOCK_N, _ptr(workspace),
        workspace.numel() * workspace.element_size(), ctypes.byref(out), _stream(stream)),
        "attn_block_mask_build")
    return BlockMask(out, workspace, (cu_seqlens, seg_id, role, turn, dense_bits, dense_offsets))


def attn_block_mask_build_noalloc(kind, cu_seqlens: torch.Tensor, total_tokens: int,
                                  max_seqlen: int, workspace: torch.Tensor,
                                  seg_id: Optional[torch.Tensor] = None,
                                  role: Optional[torch.Tensor] = None,
                                  turn: Optional[torch.Tensor] = None, role_think: int = 1,
                                  stream=None, dense_bits: Optional[torch.Tensor] = None,
                                  dense_offsets: Optional[torch.Tensor] = None) -> BlockMask:
    """Block-mask build that allocates nothing, for callers that cannot.

    The caller passes the output buffer ``workspace`` (at least
    ``attn_block_mask_workspace_size`` bytes); the builder's temporaries use a
    fixed 4 MiB array inside the library, shared by every call on the device,
    so calls must not overlap on the GPU.  The first call on a device does a
    one-time address lookup and should come before any stream capture.  Only
    the arrays the forward and backward read are stored (``labels``, ``qt_off``
    and ``pair_off`` are not).  The scratch serves up to 259,968 tokens in
    one sequence (2031 tiles); larger problems are refused.
    """
    _need_meta("attn_block_mask_build_noalloc", cu_seqlens, seg_id, role, turn, dense_bits,
               dense_offsets)
    _need(workspace, "workspace", "attn_block_mask_build_noalloc", device=cu_seqlens.device)
    batch = cu_seqlens.numel() - 1
    params = _params(role_think, dense_bits, dense_offsets)
    out = _native.AttnBlockMask()
    _check(_native.lib().attn_block_mask_build_noalloc(
        _kind(kind), ctypes.byref(params), _ptr(cu_seqlens), batch, total_tokens, max_seqlen,
        _ptr(seg_id), _ptr(role), _ptr(turn), BLOCK_M, BLOCK_N, _ptr(workspace),
        workspace.numel() * workspace.element_size(), ctypes.byref(out), _stream(stream)),
        "attn_block_mask_build_noalloc")
    return BlockMask(out, workspace, (cu_seqlens, seg_id, role, turn, dense_bits, dense_offsets),
                     noalloc=True)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, bm: BlockMask, kind,
             cu_seqlens: torch.Tensor, max_seqlen: int, seg_id=None, role=None, turn=None,
             role_think: int = 1, scale: float = 0.0, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, stream=None,
             dense_bits: Optional[torch.Tensor] = None, dense_offsets: Optional[torch.Tensor] = None):
    """Masked attention forward; returns (O [T, H, D], LSE [H, T] fp32)."""
    where = "attn_fwd"
    _need(q, "q", where, tuple(DTYPES))
    if q.dim() != 3:
        raise AttnError(1, f"{where}: q must be [T, H, D]")
    T, H, D = q.shape
    for name, t in (("k", k), ("v", v), ("out", out)):
        _need(t, name, where, (q.dtype,), q.shape, q.device)
    _need(lse, "lse", where, (torch.float32,), (H, T), q.device)
    _need_meta(where, cu_seqlens, seg_id, role, turn, dense_bits, dense_offsets, q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    params = _params(role_think, dense_bits, dense_offsets)
    _check(_native.lib().attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), DTYPES[q.dtype], T, H, D, float(scale),
        _ptr(cu_seqlens), cu_seqlens.numel() - 1, max_seqlen, _kind(kind), ctypes.byref(params),
        _ptr(seg_id), _ptr(role), _ptr(turn), ctypes.byref(bm.struct), _stream(stream)),
        "attn_fwd")
    return out, lse


def attn_bwd_workspace_size(bm: BlockMask, num_heads: int, head_dim: int) -> int:
    """Bytes of device workspace attn_bwd needs: D and ||dO_i|| per row and
    head, per-sequence bound words and the int32 fixed-point dQ accumulator,
    O(T H D)."""
    out = ctypes.c_size_t()
    _check(_native.lib().attn_bwd_workspace_size(ctypes.byref(bm.struct), num_heads, head_dim,
                                                 ctypes.byref(out)), "attn_bwd_workspace_size")
    return int(out.value)


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             lse: torch.Tensor, dout: torch.Tensor, bm: BlockMask, kind, cu_seqlens: torch.Tensor,
             max_seqlen: int, seg_id=None, role=None, turn=None, role_think: int = 1,
             scale: float = 0.0, dq: Optional[torch.Tensor] = None,
             dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, stream=None,
             dense_bits: Optional[torch.Tensor] = None, dense_offsets: Optional[torch.Tensor] = None):
    """Masked attention backward (bf16); returns (dQ, dK, dV), each [T, H, D].

    ``workspace`` (uint8, device) defaults to a fresh buffer of
    attn_bwd_workspace_size(bm, H, D) bytes.
    """
    where = "attn_bwd"
    _need(q, "q", where, tuple(DTYPES))
    if q.dim() != 3:
        raise AttnError(1, f"{where}: q must be [T, H, D]")
    T, H, D = q.shape
    if q.dtype != torch.bfloat16:
        raise AttnError(2, "attn_bwd: dtype must be bfloat16")
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, name, where, (q.dtype,), q.shape, q.device)
    if o is None or dout is None or lse is None:
        raise AttnError(1, f"{where}: o, lse and dout are required")
    _need(lse, "lse", where, (torch.float32,), (H, T), q.device)
    _need(workspace, "workspace", where, device=q.device)
    _need_meta(where, cu_seqlens, seg_id, role, turn, dense_bits, dense_offsets, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_size(bm, H, D), dtype=torch.uint8, device=q.device)
    params = _params(role_think, dense_bits, dense_offsets)
    _check(_native.lib().attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        DTYPES[q.dtype], T, H, D, float(scale), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
        max_seqlen, _kind(kind), ctypes.byref(params), _ptr(seg_id), _ptr(role), _ptr(turn),
        ctypes.byref(bm.struct), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)),
        "attn_bwd")
    return dq, dk, dv


def attn_get_status(bm: BlockMask, stream=None) -> int:
    """Synchronise and return the device status code of the mask's error word."""
    return int(_native.lib().attn_get_status(ctypes.byref(bm.struct), _stream(stream)))
