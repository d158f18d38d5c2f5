"""Position-split, quantised-KV decode attention for GB300 (sm_103a).

Thin Python binding over the C ABI of ``include/qps.h``: every function here only
marshals torch tensors (device memory, pinned host memory, streams) into the ABI's
plain pointers and sizes.  All computation runs in the library's CUDA kernels; there
is no CPU or eager-PyTorch fallback, and a missing library raises at first use.

Names follow the ABI without its ``qps_`` prefix (``kv_quant_q8_0``,
``kv_quant_tq3``, ``attn_decode_window``, ``attn_decode_tail``, ``lse_combine``,
``Ring`` for ``qps_ring_*``, ``StepPlan`` for ``qps_decode_step``).
"""

from __future__ import annotations

import ctypes
import dataclasses
from typing import List, Optional, Sequence

import torch

from . import _native as N
from ._native import FMT_F16, FMT_Q8_0, FMT_TQ2, FMT_TQ3, FMT_TQ4, QpsError  # noqa: F401

__all__ = [
    "QpsError",
    "KV",
    "tq3_codebook",
    "tq_codebook",
    "kv_quant_q8_0",
    "kv_quant_tq3",
    "plane_row_bytes",
    "Rotation",
    "kv_quant_tq2",
    "kv_quant_tq4",
    "encode_kv",
    "encode_kv_head_major",
    "attn_args",
    "attn_plan",
    "attn_decode_window",
    "lse_combine",
    "HostArena",
    "copy_host",
    "Ring",
    "tile_desc",
    "StepPlan",
    "launch_count",
    "lib",
]


def lib():
    return N.load()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _sign_array(signs):
    words = [int(w) & 0xFFFFFFFF for w in (signs.tolist() if hasattr(signs, "tolist") else signs)]
    arr = (ctypes.c_uint32 * len(words))(*words)
    return arr


@dataclasses.dataclass(frozen=True)
class Rotation:
    """A TurboQuant rotation R = diag(s2) blockdiag(H_block) diag(s1) / sqrt(block):
    sign words ``signs1`` (D/32), optional ``signs2`` and the Hadamard block width
    (0 = head_dim).  Accepted wherever TurboQuant sign words are; plain sign words mean
    ``Rotation(signs)``."""

    signs1: object
    signs2: object = None
    block: int = 0


def _rotation(signs) -> Rotation:
    return signs if isinstance(signs, Rotation) else Rotation(signs)


def _tq_encode_rot(bits: int, x2, rows: int, d: int, stride: int, rot: Rotation, p0, p1, norms, stream):
    s1 = _sign_array(rot.signs1)
    s2 = _sign_array(rot.signs2) if rot.signs2 is not None else None
    N.check(lib().qps_kv_quant_tq_rot(bits, x2.data_ptr(), rows, d, stride, s1, s2, int(rot.block),
                                      p0.data_ptr(), None if p1 is None else p1.data_ptr(),
                                      norms.data_ptr(), _stream(stream)))


def launch_count(reset: bool = False) -> int:
    return int(lib().qps_launch_count(1 if reset else 0))


def device_status(reset: bool = True) -> None:
    """Raise QpsError(QPS_ERR_TIMEOUT) if a kernel's bounded wait gave up since the last
    reset (synchronous)."""
    N.check(lib().qps_device_status(1 if reset else 0))


def device_wait_record() -> List[int]:
    """The device error word and the record of the first bounded wait that gave up
    (``qps_device_wait_record``: 16 words, synchronous)."""
    arr = (ctypes.c_uint32 * 16)()
    N.check(lib().qps_device_wait_record(arr, 16))
    return list(arr)


def selftest_bounded_wait(stream=None) -> None:
    """Enqueue the library's self-test of its bounded in-kernel waits: one warp waits on
    a barrier nothing arrives on, gives up after well under a second and sets the device
    error word, so that the next ``device_status()`` raises QpsError(QPS_ERR_TIMEOUT)."""
    N.check(lib().qps_selftest_bounded_wait(_stream(stream)))


def tq3_codebook():
    """The library's fixed TQ3 codebook: (8 levels, 7 thresholds) as Python floats."""
    lv = (ctypes.c_float * 8)()
    th = (ctypes.c_float * 7)()
    N.check(lib().qps_tq3_codebook(lv, th))
    return list(lv), list(th)


def tq_codebook(bits: int):
    """The codebook of the ``bits``-bit TurboQuant tier (2, 3 or 4): (2^bits levels,
    2^bits - 1 thresholds) as Python floats."""
    n = 1 << bits if bits in (2, 3, 4) else 1
    lv = (ctypes.c_float * n)()
    th = (ctypes.c_float * max(1, n - 1))()
    N.check(lib().qps_tq_codebook(bits, lv, th))
    return list(lv), list(th)[:n - 1]


def _rows2d(x: torch.Tensor):
    if x.dtype != torch.float16 or not x.is_cuda:
        raise QpsError(N.QPS_ERR_INVALID_ARG, "input must be a CUDA float16 tensor")
    if x.stride(-1) != 1:
        raise QpsError(N.QPS_ERR_INVALID_ARG, "input's last dimension must be contiguous")
    d = x.shape[-1]
    x2 = x.reshape(-1, d)
    stride = x2.stride(0) if x2.shape[0] > 1 else d
    return x2, d, stride


def kv_quant_q8_0(x: torch.Tensor, codes=None, scales=None, stream=None):
    """Encode fp16 rows ``x[..., D]`` as q8_0: (int8 codes [..., D], fp16 scales [..., D/32])."""
    x2, d, stride = _rows2d(x)
    rows = x2.shape[0]
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (d // 32,), dtype=torch.float16, device=x.device)
    N.check(lib().qps_kv_quant_q8_0(x2.data_ptr(), rows, d, stride, codes.data_ptr(),
                                    scales.data_ptr(), _stream(stream)))
    return codes, scales


def kv_quant_tq3(x: torch.Tensor, signs, lo2=None, hi1=None, norms=None, stream=None):
    """Encode fp16 rows ``x[..., D]`` as TQ3: (2-bit plane [..., D/4] u8, 1-bit plane
    [..., D/8] u8, fp16 norms [...])."""
    x2, d, stride = _rows2d(x)
    rows = x2.shape[0]
    if lo2 is None:
        lo2 = torch.empty(x.shape[:-1] + (d // 4,), dtype=torch.uint8, device=x.device)
    if hi1 is None:
        hi1 = torch.empty(x.shape[:-1] + (d // 8,), dtype=torch.uint8, device=x.device)
    if norms is None:
        norms = torch.empty(x.shape[:-1], dtype=torch.float16, device=x.device)
    if isinstance(signs, Rotation):
        _tq_encode_rot(3, x2, rows, d, stride, signs, lo2, hi1, norms, stream)
        return lo2, hi1, norms
    sa = _sign_array(signs)
    N.check(lib().qps_kv_quant_tq3(x2.data_ptr(), rows, d, stride, sa, lo2.data_ptr(),
                                   hi1.data_ptr(), norms.data_ptr(), _stream(stream)))
    return lo2, hi1, norms


def _kv_quant_fields(bits: int, x: torch.Tensor, signs, codes=None, norms=None, stream=None):
    x2, d, stride = _rows2d(x)
    rows = x2.shape[0]
    if codes is None:
        codes = torch.empty(x.shape[:-1] + (d * bits // 8,), dtype=torch.uint8, device=x.device)
    if norms is None:
        norms = torch.empty(x.shape[:-1], dtype=torch.float16, device=x.device)
    if isinstance(signs, Rotation):
        _tq_encode_rot(bits, x2, rows, d, stride, signs, codes, None, norms, stream)
        return codes, norms
    sa = _sign_array(signs)
    fn = lib().qps_kv_quant_tq2 if bits == 2 else lib().qps_kv_quant_tq4
    N.check(fn(x2.data_ptr(), rows, d, stride, sa, codes.data_ptr(), norms.data_ptr(), _stream(stream)))
    return codes, norms


def kv_quant_tq2(x: torch.Tensor, signs, codes=None, norms=None, stream=None):
    """Encode fp16 rows ``x[..., D]`` as TQ2: (2-bit sign-magnitude fields [..., D/4] u8,
    fp16 norms [...])."""
    return _kv_quant_fields(2, x, signs, codes, norms, stream)


def kv_quant_tq4(x: torch.Tensor, signs, codes=None, norms=None, stream=None):
    """Encode fp16 rows ``x[..., D]`` as TQ4: (4-bit sign-magnitude fields [..., D/2] u8,
    fp16 norms [...])."""
    return _kv_quant_fields(4, x, signs, codes, norms, stream)


def plane_row_bytes(fmt: str, d: int) -> List[int]:
    """Bytes per row of each stored plane of ``fmt`` (data, aux, aux2 order)."""
    return {"f16": [2 * d], "q8_0": [d, d // 16], "tq3": [d // 4, d // 8, 2],
            "tq2": [d // 4, 2], "tq4": [d // 2, 2]}[fmt]


@dataclasses.dataclass
class KV:
    """A stored K or V cache: its format, its planes and how rows are addressed.

    Planes are token-major tensors ``[(batch,) tokens, hkv, plane_row]``; the row of
    (token t, KV head h, batch entry b) is b*batch_stride + t*tok_stride + h*head_stride.
    """

    fmt: str
    planes: tuple
    tokens: int
    hkv: int
    d: int
    tok_stride: int
    head_stride: int = 1
    batch_stride: int = 0

    def view(self) -> N.KvView:
        ptrs = [p.data_ptr() for p in self.planes] + [None] * (3 - len(self.planes))
        return N.KvView(N.FMT_BY_NAME[self.fmt], 0, ptrs[0], ptrs[1], ptrs[2],
                        self.tok_stride, self.head_stride, self.batch_stride)

    def nbytes(self) -> int:
        return sum(p.numel() * p.element_size() for p in self.planes)

    def token_slice(self, t0: int, t1: int) -> "KV":
        """The positions [t0, t1) of a token-major, unbatched cache (a view, no copy)."""
        return KV(self.fmt, tuple(p[t0:t1] for p in self.planes), t1 - t0, self.hkv, self.d,
                  self.tok_stride, self.head_stride, self.batch_stride)

    def pinned_copy(self) -> "KV":
        """The same planes copied to pinned host memory."""
        planes = tuple(p.detach().to("cpu").pin_memory() for p in self.planes)
        return dataclasses.replace(self, planes=planes)


def encode_kv(fmt: str, x: torch.Tensor, signs=None, stream=None) -> KV:
    """Store fp16 ``x[(batch,) tokens, hkv, D]`` (CUDA) in ``fmt`` with the library's
    encoders; the result is token-major."""
    d = x.shape[-1]
    hkv = x.shape[-2]
    tokens = x.shape[-3]
    batch_stride = tokens * hkv if x.dim() == 4 else 0
    if fmt == "f16":
        planes = (x.contiguous(),)
    elif fmt == "q8_0":
        planes = kv_quant_q8_0(x.contiguous(), stream=stream)
    elif fmt in ("tq2", "tq3", "tq4"):
        if signs is None:
            raise QpsError(N.QPS_ERR_INVALID_ARG, "TurboQuant formats need the sign words")
        enc = {"tq2": kv_quant_tq2, "tq3": kv_quant_tq3, "tq4": kv_quant_tq4}[fmt]
        planes = enc(x.contiguous(), signs, stream=stream)
    else:
        raise QpsError(N.QPS_ERR_INVALID_ARG, f"unknown format {fmt}")
    return KV(fmt, tuple(planes), tokens, hkv, d, hkv, 1, batch_stride)


def attn_args(q: torch.Tensor, k: KV, v: KV, *, scale: float, softcap: float = 0.0,
              kv_begin: int = 0, kv_end: Optional[int] = None, v_signs=None, n_split: int = 0,
              shared: bool = False, q_pos: Optional[int] = None) -> N.AttnArgs:
    """Build the ABI argument struct for ``q[batch, hq, D]`` against (k, v).

    A 4-D ``q[batch, n_q, hq, D]`` asks for multi-query (verify-batch) decode: n_q
    query tokens per batch entry, output rows ordered (batch, token, head).  With
    ``q_pos``, query token i sees only the positions <= q_pos + i (causal).
    ``shared`` makes every batch entry read the same KV rows (batch_stride 0).
    ``v_signs``: a TurboQuant V's sign words or ``Rotation``.  The returned struct keeps
    a reference to the sign arrays it points to.
    """
    if q.dtype != torch.float16 or q.dim() not in (3, 4):
        raise QpsError(N.QPS_ERR_INVALID_ARG, "q must be float16 [batch, hq, D] or [batch, n_q, hq, D]")
    if q.dim() == 3:
        batch, hq, d = q.shape
        n_q = 1
    else:
        batch, n_q, hq, d = q.shape
        if q.stride(1) != hq * d or q.stride(2) != d or q.stride(3) != 1:
            raise QpsError(N.QPS_ERR_INVALID_ARG, "q [batch, n_q, hq, D] must be contiguous per batch entry")
    a = N.AttnArgs()
    a._tensors = (q, k, v)  # the struct holds raw pointers: keep what they point to alive
    a.q = q.data_ptr()
    a.q_batch_stride = q.stride(0)
    a.batch, a.hq, a.hkv, a.d = batch, hq, k.hkv, d
    a.n_q = n_q
    if q_pos is not None:
        a.causal, a.q_pos = 1, q_pos
    a.k = k.view()
    a.v = v.view()
    if shared:
        a.k.batch_stride = 0
        a.v.batch_stride = 0
    a.kv_begin = kv_begin
    a.kv_end = k.tokens if kv_end is None else kv_end
    a.scale = scale
    a.softcap = softcap
    if v_signs is not None:
        rot = _rotation(v_signs)
        arr = _sign_array(rot.signs1)
        a.v_signs = ctypes.cast(arr, ctypes.POINTER(ctypes.c_uint32))
        keep = [arr]
        if rot.signs2 is not None:
            arr2 = _sign_array(rot.signs2)
            a.v_signs2 = ctypes.cast(arr2, ctypes.POINTER(ctypes.c_uint32))
            keep.append(arr2)
        a.v_block = int(rot.block)
        a._keep = keep
    a.n_split = n_split
    return a


def attn_plan(a: N.AttnArgs):
    """(n_split, workspace_bytes) the library resolves for these args."""
    n = ctypes.c_int32()
    ws = ctypes.c_size_t()
    N.check(lib().qps_attn_plan(ctypes.byref(a), ctypes.byref(n), ctypes.byref(ws)))
    return n.value, ws.value


def attn_path(a: N.AttnArgs) -> str:
    """"tensor-core" or "cuda-core": the kernel the library selects for these args."""
    r = int(lib().qps_attn_path(ctypes.byref(a)))
    if r < 0:
        N.check(-r)
    return "tensor-core" if r == 1 else "cuda-core"


def attn_decode_window(a: N.AttnArgs, *, o=None, lse=None, parts=None, part_offset: int = 0,
                       workspace=None, stream=None, device=None):
    """Run one device-resident attention part.

    With ``parts=(o_parts, lse_parts)`` the split partials are written at
    ``part_offset``; otherwise the merged (o, lse) are returned (allocated if None).
    """
    rows = a.batch * max(1, a.n_q) * a.hq
    if parts is not None:
        a.o_parts, a.lse_parts = parts[0].data_ptr(), parts[1].data_ptr()
        a.part_offset = part_offset
        a.o = a.lse = None
        N.check(lib().qps_attn_decode_window(ctypes.byref(a), _stream(stream)))
        return parts
    dev = device or torch.device("cuda", torch.cuda.current_device())
    if o is None:
        o = torch.empty((rows, a.d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    a.o_parts = a.lse_parts = None
    _, ws = attn_plan(a)
    if workspace is None or workspace.numel() < ws:
        workspace = torch.empty((max(ws, 256),), dtype=torch.uint8, device=dev)
    a.o, a.lse = o.data_ptr(), lse.data_ptr()
    a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel()
    N.check(lib().qps_attn_decode_window(ctypes.byref(a), _stream(stream)))
    return o, lse


def attn_decode_window_noalloc(a: N.AttnArgs, o: torch.Tensor, lse: torch.Tensor, stream=None):
    """Merged-output decode attention that allocates no device memory: the split
    partials go to the library's fixed device scratch instead of a workspace.  For
    callers that cannot allocate on the call path; ``o`` [batch*n_q*hq, D] and ``lse``
    [batch*n_q*hq] (f32, CUDA, contiguous) must be given.  Calls sharing a device must
    not overlap."""
    rows = a.batch * max(1, a.n_q) * a.hq
    for t, n, what in ((o, rows * a.d, "o"), (lse, rows, "lse")):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.numel() != n:
            raise QpsError(N.QPS_ERR_INVALID_ARG,
                           f"attn_decode_window_noalloc: {what} must be a contiguous f32 CUDA tensor of "
                           f"{n} elements (batch*n_q*hq rows)")
    a.o_parts = a.lse_parts = None
    a.o, a.lse = o.data_ptr(), lse.data_ptr()
    a.workspace, a.workspace_bytes = None, 0
    N.check(lib().qps_attn_decode_window_noalloc(ctypes.byref(a), _stream(stream)))
    return o, lse


def lse_combine(o_parts: torch.Tensor, lse_parts: torch.Tensor, o=None, lse=None, stream=None):
    """Merge ``o_parts[P, rows, D]`` / ``lse_parts[P, rows]`` (f32, CUDA)."""
    p, rows, d = o_parts.shape
    if o is None:
        o = torch.empty((rows, d), dtype=torch.float32, device=o_parts.device)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=o_parts.device)
    N.check(lib().qps_lse_combine(o_parts.data_ptr(), lse_parts.data_ptr(), p, rows, d,
                                  o.data_ptr(), lse.data_ptr(), _stream(stream)))
    return o, lse


def encode_kv_head_major(fmt: str, x: torch.Tensor, signs=None, pad: int = 16, stream=None) -> KV:
    """Store fp16 ``x[(batch,) tokens, hkv, D]`` (CUDA) in ``fmt``, head-major: planes
    ``[(batch,) hkv, tokens_pad, row]`` with tokens_pad = tokens rounded up to ``pad``
    (the padding rows hold zeros and are never attended).  Consecutive positions of a
    head are adjacent rows, the layout the tensor-core decode streams."""
    batched = x.dim() == 4
    xb = x if batched else x.unsqueeze(0)
    b, tokens, hkv, d = xb.shape
    tp = (tokens + pad - 1) // pad * pad
    xt = torch.zeros((b, hkv, tp, d), dtype=x.dtype, device=x.device)
    xt[:, :, :tokens] = xb.permute(0, 2, 1, 3)
    kv = encode_kv(fmt, xt.reshape(b, hkv * tp, 1, d), signs, stream)
    planes = tuple(p.reshape((b, hkv, tp) + tuple(p.shape[3:])) if batched
                   else p.reshape((hkv, tp) + tuple(p.shape[3:])) for p in kv.planes)
    return KV(fmt, planes, tokens, hkv, d, tok_stride=1, head_stride=tp,
              batch_stride=hkv * tp if batched else 0)


def tile_desc(k_host: KV, v_host: KV, t0: Optional[int] = None, t1: Optional[int] = None,
              pos0: int = 0) -> N.TileDesc:
    """Ring descriptor of a pinned host tile.

    With ``t0, t1`` given, a token-major cache (row = token * hkv + head) is sliced to
    positions [t0, t1).  Without them, the cache is one whole tile described as it is
    stored (e.g. head-major, ``encode_kv_head_major``).  ``pos0``: the position of the
    tile's first token in the coordinates of a causal q_pos.
    """
    td = N.TileDesc()
    td.pos0 = int(pos0)
    if t0 is None:
        if (v_host.tok_stride, v_host.head_stride) != (1, k_host.head_stride):
            raise QpsError(N.QPS_ERR_INVALID_ARG, "K and V of a tile need the same layout")
        td.tokens = k_host.tokens
        td.tok_stride, td.head_stride = 1, k_host.head_stride
        for side, kv in (("k", k_host), ("v", v_host)):
            hosts = getattr(td, "host_" + side)
            sizes = getattr(td, "bytes_" + side)
            for i, p in enumerate(kv.planes):
                hosts[i] = p.data_ptr()
                sizes[i] = p.numel() * p.element_size()
            setattr(td, "n_%s_planes" % side, len(kv.planes))
        return td
    for kv in (k_host, v_host):
        if (kv.tok_stride, kv.head_stride, kv.batch_stride) != (kv.hkv, 1, 0):
            raise QpsError(N.QPS_ERR_INVALID_ARG, "slicing needs an unbatched token-major cache")
    td.tokens = t1 - t0
    td.tok_stride, td.head_stride = k_host.hkv, 1
    for side, kv in (("k", k_host), ("v", v_host)):
        hosts = getattr(td, "host_" + side)
        sizes = getattr(td, "bytes_" + side)
        for i, p in enumerate(kv.planes):
            row_bytes = p[0].numel() * p.element_size() if p.shape[0] > 0 else 0
            hosts[i] = p.data_ptr() + t0 * row_bytes
            sizes[i] = (t1 - t0) * row_bytes
        setattr(td, "n_%s_planes" % side, len(kv.planes))
    return td


class HostArena:
    """One page-locked host region from ``qps_host_alloc``, handed out as 256-byte
    aligned CPU tensors that alias it (no copies).  Owned until ``close()``."""

    def __init__(self, nbytes: int, flags: int = 0):
        """``flags`` as ``qps_host_alloc``: 0 cudaHostAlloc, 1 write-combined, 2 huge-page
        backed mapping registered with CUDA."""
        p = ctypes.c_void_p()
        N.check(lib().qps_host_alloc(max(int(nbytes), 256), int(flags), ctypes.byref(p)))
        self.ptr = p.value
        self.nbytes = max(int(nbytes), 256)
        self.used = 0
        self._buf = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        self.tensor = torch.frombuffer(self._buf, dtype=torch.uint8)

    def take(self, shape, dtype) -> torch.Tensor:
        n = 1
        for s in shape:
            n *= int(s)
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        off = (self.used + 255) // 256 * 256
        if off + nbytes > self.nbytes:
            raise QpsError(N.QPS_ERR_INVALID_ARG, "host arena exhausted")
        self.used = off + nbytes
        return self.tensor[off:off + nbytes].view(dtype).view(tuple(shape))

    def copy_in(self, kv: "KV") -> "KV":
        """A copy of ``kv`` (any device) whose planes live in this arena."""
        planes = []
        for p in kv.planes:
            dst = self.take(p.shape, p.dtype)
            dst.copy_(p)
            planes.append(dst)
        return dataclasses.replace(kv, planes=tuple(planes))

    def close(self):
        if self.ptr:
            self.tensor = None
            self._buf = None
            N.check(lib().qps_host_free(self.ptr))
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def copy_host(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """``qps_copy_host``: copy ``src`` into ``dst`` (same byte size, contiguous) where one
    is a CUDA tensor and the other a CPU tensor inside a ``HostArena`` (qps_host_alloc
    memory), by SM loads and stores on ``stream`` instead of the copy engine."""
    for t, what in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous():
            raise QpsError(N.QPS_ERR_INVALID_ARG, f"copy_host: {what} must be contiguous")
    if dst.is_cuda == src.is_cuda:
        raise QpsError(N.QPS_ERR_INVALID_ARG, "copy_host: one of dst / src must be a CUDA tensor, the other host")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise QpsError(N.QPS_ERR_INVALID_ARG, "copy_host: dst and src differ in size")
    N.check(lib().qps_copy_host(dst.data_ptr(), src.data_ptr(), nbytes, _stream(stream)))
    return dst


RING_COPY = {"engine": 0, "kernel": 1}  # QPS_RING_COPY_ENGINE / QPS_RING_COPY_KERNEL


class Ring:
    """The tail-prefetch ring (``qps_ring_*``): device staging slots, a copy stream and
    pre-created copy_done / compute_done events, owned by the library."""

    def __init__(self, n_slots: int, slot_bytes: int, device: Optional[int] = None, copy: str = "engine"):
        """``copy``: "engine" (cudaMemcpyAsync) or "kernel" (the ring's copy kernel for
        tiles in ``HostArena`` / qps_host_alloc memory, the copy engine otherwise)."""
        dev = torch.cuda.current_device() if device is None else device
        h = ctypes.c_void_p()
        N.check(lib().qps_ring_create(n_slots, slot_bytes, dev, ctypes.byref(h)))
        self.handle = h
        self.n_slots = n_slots
        self.slot_bytes = slot_bytes
        self._tiles = None
        if copy not in RING_COPY:
            raise QpsError(N.QPS_ERR_INVALID_ARG, f"unknown ring copy mode {copy}")
        N.check(lib().qps_ring_set_copy_mode(self.handle, RING_COPY[copy]))

    def begin_step(self, tiles: Sequence[N.TileDesc], stream=None):
        arr = (N.TileDesc * len(tiles))(*tiles)
        self._tiles = arr
        N.check(lib().qps_ring_begin_step(self.handle, arr, len(tiles), _stream(stream)))

    def decode_tail(self, index: int, a: N.AttnArgs, *, parts, part_offset: int, stream=None):
        a.o_parts, a.lse_parts = parts[0].data_ptr(), parts[1].data_ptr()
        a.part_offset = part_offset
        N.check(lib().qps_attn_decode_tail(self.handle, index, ctypes.byref(a), _stream(stream)))

    def end_step(self):
        N.check(lib().qps_ring_end_step(self.handle))

    def sync(self, timeout_ms: int = 10000):
        N.check(lib().qps_ring_sync(self.handle, timeout_ms))

    def check_guards(self, timeout_ms: int = 10000) -> None:
        """Wait for the ring's work, then compare the guard regions around every slot
        with their pattern (``qps_ring_check_guards``); raises QpsError(INTERNAL) if
        something wrote outside a slot."""
        bad = ctypes.c_int32(-1)
        N.check(lib().qps_ring_check_guards(self.handle, timeout_ms, ctypes.byref(bad)))

    def slot(self, index: int):
        """(device address, usable bytes) of slot ``index``."""
        p, n = ctypes.c_void_p(), ctypes.c_size_t()
        N.check(lib().qps_ring_slot(self.handle, index, ctypes.byref(p), ctypes.byref(n)))
        return p.value, n.value

    FAULTS = {"none": 0, "copy_fail": 1, "copy_late": 2}

    def inject_fault(self, tile_index: int, mode: str, delay_ms: int = 0) -> None:
        """Arm a one-shot host-side fault on the next copy of schedule index
        ``tile_index`` (``qps_ring_inject_fault``): "copy_fail", "copy_late" or "none"."""
        N.check(lib().qps_ring_inject_fault(self.handle, tile_index, self.FAULTS[mode], delay_ms))

    def close(self):
        if self.handle:
            N.check(lib().qps_ring_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepPlan:
    """A whole decode step prepared once and run with one ``qps_decode_step`` call.

    ``layers`` is a list of dicts with keys ``device_parts`` (list of AttnArgs),
    ``tail`` (AttnArgs or None), ``n_tiles``, ``o_parts``, ``lse_parts`` (f32 CUDA
    tensors [capacity, rows, D] / [capacity, rows]), ``o``, ``lse`` and optionally
    ``part_events`` (two raw cudaEvent_t handles recorded around the device parts).
    """

    def __init__(self, layers: List[dict], tiles: Sequence[N.TileDesc] = (), ring: Optional[Ring] = None):
        self.ring = ring
        self.tiles = (N.TileDesc * max(1, len(tiles)))(*tiles)
        self.n_tiles = len(tiles)
        self._keep = []
        steps = []
        for L in layers:
            parts = (N.AttnArgs * max(1, len(L["device_parts"])))(*L["device_parts"])
            tail = L.get("tail")
            tail_ptr = None
            if tail is not None:
                tail_arr = (N.AttnArgs * 1)(tail)
                tail_ptr = ctypes.cast(tail_arr, ctypes.POINTER(N.AttnArgs))
                self._keep.append(tail_arr)
            self._keep += [parts, L["device_parts"], tail]
            st = N.LayerStep()
            st.device_parts = ctypes.cast(parts, ctypes.POINTER(N.AttnArgs))
            st.n_device_parts = len(L["device_parts"])
            st.n_tiles = L.get("n_tiles", 0)
            st.tail = tail_ptr
            st.o_parts = L["o_parts"].data_ptr()
            st.lse_parts = L["lse_parts"].data_ptr()
            st.parts_capacity = L["o_parts"].shape[0]
            st.o = L["o"].data_ptr()
            st.lse = L["lse"].data_ptr()
            ev = L.get("part_events")
            if ev is not None:
                st.part_events[0], st.part_events[1] = ev
            steps.append(st)
        self.layers = (N.LayerStep * len(steps))(*steps)
        self.n_layers = len(steps)

    def run(self, stream=None):
        ring = self.ring.handle if self.ring is not None else None
        N.check(lib().qps_decode_step(ring, self.tiles, self.n_tiles, self.layers, self.n_layers,
                                      _stream(stream)))


# ---- residency and ring sizing policy (host arithmetic in the library) -------------
def plan_ring(compute_ms_per_layer: float, bw_eff_gbs: float, slot_budget_bytes: float,
              per_layer_tail_bytes: float) -> dict:
    """Ring slots and tail tiling from one layer's attention time and the link
    bandwidth (``qps_plan_ring``)."""
    n, t = ctypes.c_int32(), ctypes.c_int32()
    tb, tmax = ctypes.c_double(), ctypes.c_double()
    N.check(lib().qps_plan_ring(compute_ms_per_layer, bw_eff_gbs, slot_budget_bytes, per_layer_tail_bytes,
                                ctypes.byref(n), ctypes.byref(t), ctypes.byref(tb), ctypes.byref(tmax)))
    return {"n_slots": n.value, "tiles_per_layer": t.value, "tile_bytes": tb.value, "tile_bytes_max": tmax.value}


def tail_band(t_resident_ms: float, c_engage_ms: float, bw_eff_gbs: float, target_drop: float = 0.20) -> float:
    """T*: the largest streamed tail (bytes) within ``target_drop`` (``qps_tail_band``)."""
    out = ctypes.c_double()
    N.check(lib().qps_tail_band(t_resident_ms, c_engage_ms, bw_eff_gbs, target_drop, ctypes.byref(out)))
    return out.value


def choose_tier(kv_bytes_per_tier, budget_bytes: float, t_star_bytes: float) -> int:
    """The first storage tier whose bytes fit budget + T* (``qps_choose_tier``)."""
    arr = (ctypes.c_double * len(kv_bytes_per_tier))(*[float(x) for x in kv_bytes_per_tier])
    out = ctypes.c_int32()
    N.check(lib().qps_choose_tier(arr, len(kv_bytes_per_tier), budget_bytes, t_star_bytes, ctypes.byref(out)))
    return out.value
