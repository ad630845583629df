"""Absorbed-latent MLA decode on GB300 (sm_103a): Python binding of libmla.so.

The binding only marshals arguments: every step of the decode path runs in the
library's CUDA kernels (see ``include/mla.h``). PyTorch provides device memory
and the current stream. There is no fallback: if the library is not built or
the GPU is not an sm_103 part, the calls raise.

The four calls of the decode path, in order:
  append_latent -> cache rows [c_kv | RoPE(k_rope)]     (576 bf16 per token)
  absorb_q      -> q_abs = [W_UK^T q_nope | RoPE(q_rope)]
  decode_attn   -> o_lat = softmax(scale q_abs . row) . c_kv, lse
  expand_v      -> out = W_UV o_lat
"""
from __future__ import annotations

import ctypes
import math
import os

from ._build import LIB, build  # noqa: F401

D_NOPE, D_ROPE, D_C, D_V = 128, 64, 512, 128
ROW = D_C + D_ROPE
ROW8 = 656          # FP8 cache row: e4m3 latent (512) | bf16 RoPE key (128) | fp32 scale | 12 zero bytes
BLOCK = 64
DEFAULT_SCALE = 1.0 / math.sqrt(D_NOPE + D_ROPE)

DEVICE_BOUNDS = 1
DEVICE_TIMEOUT = 2
DEVICE_LENGTH = 4

_STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
           4: "MLA_ERR_TIMEOUT", 5: "MLA_ERR_BOUNDS"}

# Every exported symbol of include/mla.h with its ctypes signature.
_c_void_p, _i32, _sz, _f32, _u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float, ctypes.c_uint64


class CacheDesc(ctypes.Structure):
    """mla_cache_t."""
    _fields_ = [("base", _c_void_p), ("paged", _i32), ("num_seqs", _i32), ("capacity", _i32),
                ("num_blocks", _i32), ("block_table", _c_void_p), ("max_blocks", _i32)]


SIGNATURES = {
    "mla_create": (_i32, [ctypes.POINTER(_c_void_p), _i32, _i32, ctypes.c_double]),
    "mla_destroy": (_i32, [_c_void_p]),
    "mla_last_error": (ctypes.c_char_p, [_c_void_p]),
    "mla_num_sms": (_i32, [_c_void_p]),
    "mla_append_latent": (_i32, [_c_void_p, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _c_void_p,
                                 _c_void_p, _i32, _c_void_p]),
    "mla_absorb_q": (_i32, [_c_void_p, _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32,
                            _c_void_p, _c_void_p]),
    "mla_append_latent_fp8": (_i32, [_c_void_p, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _c_void_p,
                                     _c_void_p, _i32, _c_void_p]),
    "mla_decode_attn_fp8": (_i32, [_c_void_p, _i32, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _i32, _i32,
                                   _f32, _c_void_p, _sz, _c_void_p, _c_void_p, _c_void_p]),
    "mla_append_absorb_q": (_i32, [_c_void_p, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                   _i32, _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _c_void_p,
                                   _c_void_p]),
    "mla_append_fp8_absorb_q": (_i32, [_c_void_p, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _c_void_p,
                                       _c_void_p, _i32, _i32, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32,
                                       _c_void_p, _c_void_p]),
    "mla_decode_workspace_size": (_sz, [_c_void_p, _i32, _i32, _i32]),
    "mla_decode_attn": (_i32, [_c_void_p, _i32, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _i32, _i32,
                               _f32, _c_void_p, _sz, _c_void_p, _c_void_p, _c_void_p]),
    "mla_expand_v": (_i32, [_c_void_p, _i32, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _c_void_p]),
    "mla_out_proj": (_i32, [_c_void_p, _i32, _c_void_p, _i32, _c_void_p, _i32, _c_void_p, _c_void_p]),
    "mla_project_latent_workspace_size": (ctypes.c_size_t, [_i32]),
    "mla_project_latent": (_i32, [_c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, ctypes.c_float, _c_void_p,
                                  _c_void_p, _c_void_p, _i32, _c_void_p, ctypes.c_size_t, _c_void_p]),
    "mla_small_step_max_len": (_sz, []),
    "mla_decode_step_small": (_i32, [_c_void_p, _i32, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _c_void_p,
                                     _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _f32, _c_void_p, _c_void_p,
                                     _c_void_p, _c_void_p]),
    "mla_absorb_w_o": (_i32, [_c_void_p, _i32, _c_void_p, _i32, _c_void_p, _c_void_p, _c_void_p]),
    "mla_out_proj_latent": (_i32, [_c_void_p, _i32, _c_void_p, _i32, _c_void_p, _i32, _c_void_p, _c_void_p]),
    "mla_get_device_status": (_i32, [_c_void_p, _c_void_p, ctypes.POINTER(_i32)]),
    "mla_set_decode_units": (_i32, [_c_void_p, _i32]),
    "mla_debug_wait_timeout": (_i32, [_c_void_p, _u64, _c_void_p]),
    "mla_copy_async": (_i32, [_c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "mla_decode_attn_static_scratch": (_i32, [_c_void_p, _i32, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p,
                                              _i32, _i32, _f32, _c_void_p, _c_void_p, _c_void_p]),
    "mla_static_scratch_bytes": (_sz, []),
    "mla_prefill_mha_workspace_size": (_sz, [_i32, _i32, _i32, _i32]),
    "mla_prefill_mha": (_i32, [_c_void_p, _i32, ctypes.POINTER(CacheDesc), _c_void_p, _c_void_p, _c_void_p,
                               _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _f32, _c_void_p, _sz,
                               _c_void_p, _c_void_p]),
    "mla_prefill_choose_form": (_i32, [_i32, _i32, _i32, ctypes.POINTER(ctypes.c_int32), _i32, _sz,
                                       ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)]),
}

_lib = None


class MLAError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{_STATUS.get(code, code)}: {msg}")
        self.code = code


def load_library(path: str = LIB):
    """Load libmla.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with mla_absorbed_latent_02_gb300.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _torch():
    import torch
    return torch


def _ptr(t, dtype=None, name="tensor"):
    torch = _torch()
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _out_ptr(t, dtype, name):
    """An output the kernels write with plain stores: a CUDA tensor, or pinned
    host memory (which the device addresses directly under unified addressing;
    on a coherent host link the result then reaches the host without a copy)."""
    if t is not None and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous() or t.dtype != dtype:
            raise ValueError(f"{name} must be contiguous {dtype}")
        return ctypes.c_void_p(t.data_ptr())
    return _ptr(t, dtype, name)


def _any_ptr(t, name):
    """A contiguous CUDA tensor or pinned host tensor (device-addressable)."""
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    return ctypes.c_void_p(t.data_ptr())


PREFILL_FORMS = {0: "absorbed", 1: "mha"}


def prefill_choose_form(H: int, T: int, seq_lens, fp8: bool = False, ws_limit: int = 0):
    """Which form of a prefill chunk of T new tokens per sequence to run
    (mla_prefill_choose_form, host only): returns ("absorbed" | "mha",
    (estimated µs per step of the absorbed form, of the MHA form))."""
    lens = [int(x) for x in seq_lens]
    arr = (ctypes.c_int32 * max(1, len(lens)))(*lens)
    form = ctypes.c_int32(-1)
    est = (ctypes.c_double * 2)()
    rc = load_library().mla_prefill_choose_form(H, len(lens), T, arr, int(bool(fp8)), ws_limit, ctypes.byref(form),
                                                est)
    if rc != 0:
        raise MLAError(rc, f"prefill_choose_form(H={H}, T={T}, B={len(lens)}) rejected")
    return PREFILL_FORMS[form.value], (est[0], est[1])


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Cache:
    """A latent cache in device memory: contiguous [B, capacity, 576] or paged
    [num_blocks, 64, 576] with an int32 block table [B, max_blocks]. With
    ``fp8=True`` the rows are the 656-byte FP8 rows (uint8 storage
    [..., 656]); append_latent and decode_attn then use the FP8 calls."""

    def __init__(self, storage, paged: bool, num_seqs: int, capacity: int = 0, block_table=None,
                 fp8: bool = False):
        torch = _torch()
        self.fp8 = bool(fp8)
        if self.fp8:
            if storage.dtype != torch.uint8 or storage.shape[-1] != ROW8:
                raise ValueError("FP8 cache storage must be uint8 with rows of 656 bytes")
        elif storage.dtype != torch.bfloat16 or storage.shape[-1] != ROW:
            raise ValueError("cache storage must be bf16 with rows of 576")
        self.storage = storage
        self.paged = bool(paged)
        self.num_seqs = int(num_seqs)
        self.capacity = int(capacity)
        self.block_table = block_table
        if self.paged:
            if block_table is None or block_table.dtype != torch.int32 or block_table.dim() != 2:
                raise ValueError("paged cache needs an int32 [B, max_blocks] block table")
            self.num_blocks = storage.numel() // (BLOCK * (ROW8 if self.fp8 else ROW))
            self.max_blocks = int(block_table.shape[1])
        else:
            self.num_blocks = 0
            self.max_blocks = 0
        self.desc = CacheDesc(
            ctypes.c_void_p(storage.data_ptr()), int(self.paged), self.num_seqs, self.capacity,
            self.num_blocks, ctypes.c_void_p(block_table.data_ptr()) if self.paged else None,
            self.max_blocks)

    @staticmethod
    def _storage(shape, fp8, device):
        torch = _torch()
        if fp8:
            return torch.zeros(*shape, ROW8, dtype=torch.uint8, device=device)
        return torch.zeros(*shape, ROW, dtype=torch.bfloat16, device=device)

    @staticmethod
    def contiguous(num_seqs: int, capacity: int, device="cuda", fp8: bool = False):
        st = Cache._storage((num_seqs, capacity), fp8, device)
        return Cache(st, False, num_seqs, capacity, fp8=fp8)

    @staticmethod
    def paged_pool(num_blocks: int, block_table, device="cuda", fp8: bool = False):
        torch = _torch()
        st = Cache._storage((num_blocks, BLOCK), fp8, device)
        bt = block_table.to(device=device, dtype=torch.int32).contiguous()
        return Cache(st, True, bt.shape[0], 0, bt, fp8=fp8)


class Context:
    """An mla_ctx_t: device, RoPE table (positions < max_pos) and status word."""

    def __init__(self, device: int = 0, max_pos: int = 131072, rope_base: float = 10000.0):
        self.lib = load_library()
        h = ctypes.c_void_p()
        rc = self.lib.mla_create(ctypes.byref(h), device, max_pos, rope_base)
        if rc != 0:
            raise MLAError(rc, f"mla_create(device={device}, max_pos={max_pos}) failed")
        self.h = h
        self.device = device
        self.max_pos = max_pos

    def close(self):
        if getattr(self, "h", None):
            self.lib.mla_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc):
        if rc != 0:
            raise MLAError(rc, self.lib.mla_last_error(self.h).decode())

    @property
    def num_sms(self) -> int:
        return self.lib.mla_num_sms(self.h)

    def set_decode_units(self, units: int):
        self._check(self.lib.mla_set_decode_units(self.h, units))

    def append_latent(self, cache: Cache, c_kv, k_rope, seq_idx, pos, stream=None):
        torch = _torch()
        n = int(c_kv.shape[0])
        if tuple(c_kv.shape) != (n, D_C) or tuple(k_rope.shape) != (n, D_ROPE):
            raise ValueError("c_kv must be [n, 512] and k_rope [n, 64]")
        if seq_idx.numel() != n or pos.numel() != n:
            raise ValueError("seq_idx and pos must hold n entries")
        fn = self.lib.mla_append_latent_fp8 if cache.fp8 else self.lib.mla_append_latent
        self._check(fn(
            self.h, ctypes.byref(cache.desc), _ptr(c_kv, torch.bfloat16, "c_kv"),
            _ptr(k_rope, torch.bfloat16, "k_rope"), _ptr(seq_idx, torch.int32, "seq_idx"),
            _ptr(pos, torch.int32, "pos"), n, _stream(stream)))

    def absorb_q(self, w_uk, q_nope, q_rope, q_pos, q_abs=None, stream=None):
        torch = _torch()
        B, Hq, H, dn = q_nope.shape
        if dn != D_NOPE or tuple(q_rope.shape) != (B, Hq, H, D_ROPE) or tuple(w_uk.shape) != (H, D_NOPE, D_C):
            raise ValueError("shapes: q_nope [B,Hq,H,128], q_rope [B,Hq,H,64], w_uk [H,128,512]")
        if tuple(q_pos.shape) != (B, Hq):
            raise ValueError("q_pos must be [B, Hq]")
        if q_abs is None:
            q_abs = torch.empty(B, Hq, H, ROW, dtype=torch.bfloat16, device=q_nope.device)
        self._check(self.lib.mla_absorb_q(
            self.h, H, _ptr(w_uk, torch.bfloat16, "w_uk"), _ptr(q_nope, torch.bfloat16, "q_nope"),
            _ptr(q_rope, torch.bfloat16, "q_rope"), _ptr(q_pos, torch.int32, "q_pos"), B, Hq,
            _ptr(q_abs, torch.bfloat16, "q_abs"), _stream(stream)))
        return q_abs

    def append_absorb_q(self, cache: Cache, c_kv, k_rope, seq_idx, pos, w_uk, q_nope, q_rope, q_pos, q_abs=None,
                        stream=None):
        """append_latent and absorb_q in one launch; returns q_abs."""
        torch = _torch()
        n = int(c_kv.shape[0])
        if tuple(c_kv.shape) != (n, D_C) or tuple(k_rope.shape) != (n, D_ROPE):
            raise ValueError("c_kv must be [n, 512] and k_rope [n, 64]")
        if seq_idx.numel() != n or pos.numel() != n:
            raise ValueError("seq_idx and pos must hold n entries")
        B, Hq, H, dn = q_nope.shape
        if dn != D_NOPE or tuple(q_rope.shape) != (B, Hq, H, D_ROPE) or tuple(w_uk.shape) != (H, D_NOPE, D_C):
            raise ValueError("shapes: q_nope [B,Hq,H,128], q_rope [B,Hq,H,64], w_uk [H,128,512]")
        if tuple(q_pos.shape) != (B, Hq):
            raise ValueError("q_pos must be [B, Hq]")
        if q_abs is None:
            q_abs = torch.empty(B, Hq, H, ROW, dtype=torch.bfloat16, device=q_nope.device)
        fn = self.lib.mla_append_fp8_absorb_q if cache.fp8 else self.lib.mla_append_absorb_q
        self._check(fn(
            self.h, ctypes.byref(cache.desc), _ptr(c_kv, torch.bfloat16, "c_kv"),
            _ptr(k_rope, torch.bfloat16, "k_rope"), _ptr(seq_idx, torch.int32, "seq_idx"),
            _ptr(pos, torch.int32, "pos"), n, H, _ptr(w_uk, torch.bfloat16, "w_uk"),
            _ptr(q_nope, torch.bfloat16, "q_nope"), _ptr(q_rope, torch.bfloat16, "q_rope"),
            _ptr(q_pos, torch.int32, "q_pos"), B, Hq, _ptr(q_abs, torch.bfloat16, "q_abs"), _stream(stream)))
        return q_abs

    def workspace_size(self, H: int, B: int, Hq: int) -> int:
        return int(self.lib.mla_decode_workspace_size(self.h, H, B, Hq))

    def alloc_workspace(self, H, B, Hq, device="cuda"):
        torch = _torch()
        n = self.workspace_size(H, B, Hq)
        if n == 0:
            raise MLAError(1, "invalid workspace shape")
        return torch.empty((n + 3) // 4, dtype=torch.float32, device=device)

    def decode_attn(self, cache: Cache, q_abs, seq_lens, scale: float = DEFAULT_SCALE, workspace=None,
                    o_lat=None, lse=None, stream=None):
        torch = _torch()
        B, Hq, H, r = q_abs.shape
        if r != ROW:
            raise ValueError("q_abs must be [B, Hq, H, 576]")
        if seq_lens.numel() != B:
            raise ValueError("seq_lens must hold B entries")
        if workspace is None:
            workspace = self.alloc_workspace(H, B, Hq, q_abs.device)
        if o_lat is None:
            o_lat = torch.empty(B, Hq, H, D_C, dtype=torch.float32, device=q_abs.device)
        if lse is None:
            lse = torch.empty(B, Hq, H, dtype=torch.float32, device=q_abs.device)
        fn = self.lib.mla_decode_attn_fp8 if cache.fp8 else self.lib.mla_decode_attn
        self._check(fn(
            self.h, H, ctypes.byref(cache.desc), _ptr(q_abs, torch.bfloat16, "q_abs"),
            _ptr(seq_lens, torch.int32, "seq_lens"), B, Hq, float(scale), _ptr(workspace, None, "workspace"),
            workspace.numel() * workspace.element_size(), _ptr(o_lat, torch.float32, "o_lat"),
            _ptr(lse, torch.float32, "lse"), _stream(stream)))
        return o_lat, lse

    def decode_attn_static_scratch(self, cache: Cache, q_abs, seq_lens, scale: float = DEFAULT_SCALE,
                                   o_lat=None, lse=None, stream=None):
        """decode_attn without a workspace argument, for callers that cannot
        allocate device memory: the library's fixed 16 MiB device scratch holds
        the split-KV partials. Pass preallocated o_lat / lse to allocate nothing."""
        torch = _torch()
        if cache.fp8:
            raise ValueError("decode_attn_static_scratch reads bf16 caches only")
        B, Hq, H, r = q_abs.shape
        if r != ROW:
            raise ValueError("q_abs must be [B, Hq, H, 576]")
        if seq_lens.numel() != B:
            raise ValueError("seq_lens must hold B entries")
        if o_lat is None:
            o_lat = torch.empty(B, Hq, H, D_C, dtype=torch.float32, device=q_abs.device)
        if lse is None:
            lse = torch.empty(B, Hq, H, dtype=torch.float32, device=q_abs.device)
        self._check(self.lib.mla_decode_attn_static_scratch(
            self.h, H, ctypes.byref(cache.desc), _ptr(q_abs, torch.bfloat16, "q_abs"),
            _ptr(seq_lens, torch.int32, "seq_lens"), B, Hq, float(scale), _ptr(o_lat, torch.float32, "o_lat"),
            _ptr(lse, torch.float32, "lse"), _stream(stream)))
        return o_lat, lse

    def prefill_mha_workspace_size(self, H: int, B: int, T: int, max_len: int) -> int:
        return int(self.lib.mla_prefill_mha_workspace_size(H, B, T, max_len))

    def prefill_mha(self, cache: Cache, w_uk, w_uv, q_nope, q_rope, q_pos, seq_lens, max_len: int,
                    scale: float = DEFAULT_SCALE, workspace=None, out=None, stream=None):
        """Attention of a prompt chunk of T tokens per sequence in the expanded
        (MHA) form: out [B, T, H, 128] bf16 from q_nope [B, T, H, 128] and
        q_rope [B, T, H, 64] (before RoPE, rotated at q_pos [B*T]) over the
        cache, whose sequences hold seq_lens[b] tokens with the chunk last
        (T <= seq_lens[b] <= max_len)."""
        torch = _torch()
        if cache.fp8:
            raise ValueError("prefill_mha reads bf16 caches only")
        B, T, H, dn = q_nope.shape
        if dn != D_NOPE or tuple(q_rope.shape) != (B, T, H, D_ROPE):
            raise ValueError("q_nope [B,T,H,128] and q_rope [B,T,H,64]")
        if seq_lens.numel() != B or q_pos.numel() != B * T:
            raise ValueError("seq_lens must hold B entries and q_pos B*T")
        if workspace is None:
            n = self.prefill_mha_workspace_size(H, B, T, max_len)
            workspace = torch.empty((n + 15) // 16, 16, dtype=torch.uint8, device=q_nope.device)
        if out is None:
            out = torch.empty(B, T, H, D_V, dtype=torch.bfloat16, device=q_nope.device)
        self._check(self.lib.mla_prefill_mha(
            self.h, H, ctypes.byref(cache.desc), _ptr(w_uk, torch.bfloat16, "w_uk"),
            _ptr(w_uv, torch.bfloat16, "w_uv"), _ptr(q_nope, torch.bfloat16, "q_nope"),
            _ptr(q_rope, torch.bfloat16, "q_rope"), _ptr(q_pos, torch.int32, "q_pos"),
            _ptr(seq_lens, torch.int32, "seq_lens"), B, T, int(max_len), float(scale),
            _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
            _out_ptr(out, torch.bfloat16, "out"), _stream(stream)))
        return out

    def static_scratch_bytes(self) -> int:
        return int(self.lib.mla_static_scratch_bytes())

    def copy_async(self, dst, src, stream=None):
        """dst <- src (same number of bytes) by the library's copy kernel; each
        side a CUDA tensor or pinned host memory."""
        nbytes = dst.numel() * dst.element_size()
        if src.numel() * src.element_size() != nbytes:
            raise ValueError("dst and src must have the same size in bytes")
        self._check(self.lib.mla_copy_async(self.h, _any_ptr(dst, "dst"), _any_ptr(src, "src"), nbytes,
                                            _stream(stream)))
        return dst

    def expand_v(self, w_uv, o_lat, out=None, stream=None):
        """out [B,Hq,H,128] bf16 = W_UV o_lat; ``out`` may be a CUDA tensor or
        pinned host memory (written directly by the kernel)."""
        torch = _torch()
        B, Hq, H, dc = o_lat.shape
        if dc != D_C or tuple(w_uv.shape) != (H, D_V, D_C):
            raise ValueError("shapes: o_lat [B,Hq,H,512], w_uv [H,128,512]")
        if out is None:
            out = torch.empty(B, Hq, H, D_V, dtype=torch.bfloat16, device=o_lat.device)
        self._check(self.lib.mla_expand_v(
            self.h, H, _ptr(w_uv, torch.bfloat16, "w_uv"), _ptr(o_lat, torch.float32, "o_lat"), B, Hq,
            _out_ptr(out, torch.bfloat16, "out"), _stream(stream)))
        return out

    def project_latent(self, cache: "Cache", w_kv_a, h, seq_idx, pos, kv_norm=None, eps: float = 1e-6,
                       workspace=None, stream=None):
        """Cache rows of n new tokens from their hidden states h [n, d_model]:
        [RMSNorm(W_KV_A[:512] h) | RoPE_pos(W_KV_A[512:] h)] (bf16), written at
        (seq_idx, pos) like append_latent. w_kv_a [576, d_model] bf16, kv_norm
        [512] bf16 or None (no normalisation)."""
        torch = _torch()
        if cache.fp8:
            raise ValueError("project_latent writes bf16 caches only")
        n, d_model = int(h.shape[0]), int(h.shape[1])
        if tuple(w_kv_a.shape) != (ROW, d_model):
            raise ValueError("w_kv_a must be [576, d_model]")
        if workspace is None:
            nbytes = self.lib.mla_project_latent_workspace_size(n)
            workspace = torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=h.device)
        self._check(self.lib.mla_project_latent(
            self.h, ctypes.byref(cache.desc), _ptr(w_kv_a, torch.bfloat16, "w_kv_a"), d_model,
            None if kv_norm is None else _ptr(kv_norm, torch.bfloat16, "kv_norm"), float(eps),
            _ptr(h, torch.bfloat16, "h"), _ptr(seq_idx, torch.int32, "seq_idx"), _ptr(pos, torch.int32, "pos"), n,
            _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)))

    def out_proj(self, w_o, o, y=None, stream=None):
        """y [M, d_model] fp32 = W_O concat_h(o[r, h, :]) for o [..., H, 128] bf16
        (rows = all leading dimensions) and w_o [d_model, H*128] bf16."""
        torch = _torch()
        H, dv = int(o.shape[-2]), int(o.shape[-1])
        M = int(o.numel() // (H * dv))
        d_model = int(w_o.shape[0])
        if dv != D_V or tuple(w_o.shape) != (d_model, H * D_V):
            raise ValueError("shapes: o [..., H, 128], w_o [d_model, H*128]")
        if y is None:
            y = torch.empty(M, d_model, dtype=torch.float32, device=o.device)
        self._check(self.lib.mla_out_proj(
            self.h, H, _ptr(w_o, torch.bfloat16, "w_o"), d_model, _ptr(o, torch.bfloat16, "o"), M,
            _ptr(y, torch.float32, "y"), _stream(stream)))
        return y

    def decode_step_small(self, cache: Cache, c_kv, k_rope, w_uk, w_uv, q_nope, q_rope, seq_lens,
                          scale: float = DEFAULT_SCALE, out=None, o_lat=None, lse=None, stream=None):
        """The whole decode step for short sequences in one launch (append of each
        sequence's new token at position seq_lens[b] - 1, absorb_q, attention,
        expand_v); one query token per sequence. c_kv [B, 512], k_rope [B, 64],
        q_nope [B, 1 or none, H, 128], q_rope [B, ..., H, 64]; returns (out, o_lat, lse)."""
        torch = _torch()
        if cache.fp8:
            raise ValueError("decode_step_small reads bf16 caches only")
        H = int(w_uk.shape[0])
        B = int(seq_lens.numel())
        if tuple(c_kv.shape) != (B, D_C) or tuple(k_rope.shape) != (B, D_ROPE):
            raise ValueError("c_kv must be [B, 512] and k_rope [B, 64]")
        if q_nope.numel() != B * H * D_NOPE or q_rope.numel() != B * H * D_ROPE:
            raise ValueError("q_nope / q_rope must hold [B, H, 128] / [B, H, 64]")
        if tuple(w_uk.shape) != (H, D_NOPE, D_C) or tuple(w_uv.shape) != (H, D_V, D_C):
            raise ValueError("w_uk, w_uv must be [H, 128, 512]")
        dev = q_nope.device
        if out is None:
            out = torch.empty(B, 1, H, D_V, dtype=torch.bfloat16, device=dev)
        if o_lat is None:
            o_lat = torch.empty(B, 1, H, D_C, dtype=torch.float32, device=dev)
        if lse is None:
            lse = torch.empty(B, 1, H, dtype=torch.float32, device=dev)
        self._check(self.lib.mla_decode_step_small(
            self.h, H, ctypes.byref(cache.desc), _ptr(c_kv, torch.bfloat16, "c_kv"),
            _ptr(k_rope, torch.bfloat16, "k_rope"), _ptr(w_uk, torch.bfloat16, "w_uk"),
            _ptr(w_uv, torch.bfloat16, "w_uv"), _ptr(q_nope, torch.bfloat16, "q_nope"),
            _ptr(q_rope, torch.bfloat16, "q_rope"), _ptr(seq_lens, torch.int32, "seq_lens"), B, float(scale),
            _out_ptr(out, torch.bfloat16, "out"), _ptr(o_lat, torch.float32, "o_lat"),
            _ptr(lse, torch.float32, "lse"), _stream(stream)))
        return out, o_lat, lse

    def absorb_w_o(self, w_o, w_uv, w_ov=None, stream=None):
        """w_ov [d_model, H*512] bf16: W_UV folded into W_O (a one-time weight
        transform) for out_proj_latent."""
        torch = _torch()
        H = int(w_uv.shape[0])
        d_model = int(w_o.shape[0])
        if tuple(w_uv.shape) != (H, D_V, D_C) or tuple(w_o.shape) != (d_model, H * D_V):
            raise ValueError("shapes: w_o [d_model, H*128], w_uv [H,128,512]")
        if w_ov is None:
            w_ov = torch.empty(d_model, H * D_C, dtype=torch.bfloat16, device=w_o.device)
        self._check(self.lib.mla_absorb_w_o(
            self.h, H, _ptr(w_o, torch.bfloat16, "w_o"), d_model, _ptr(w_uv, torch.bfloat16, "w_uv"),
            _ptr(w_ov, torch.bfloat16, "w_ov"), _stream(stream)))
        return w_ov

    def out_proj_latent(self, w_ov, o_lat, y=None, stream=None):
        """y [M, d_model] fp32 = W_OV concat_h(o_lat[r, h, :]) for o_lat [..., H, 512]
        fp32 (rows = all leading dimensions): expand_v and out_proj in one GEMM."""
        torch = _torch()
        H, dc = int(o_lat.shape[-2]), int(o_lat.shape[-1])
        M = int(o_lat.numel() // (H * dc))
        d_model = int(w_ov.shape[0])
        if dc != D_C or tuple(w_ov.shape) != (d_model, H * D_C):
            raise ValueError("shapes: o_lat [..., H, 512], w_ov [d_model, H*512]")
        if y is None:
            y = torch.empty(M, d_model, dtype=torch.float32, device=o_lat.device)
        self._check(self.lib.mla_out_proj_latent(
            self.h, H, _ptr(w_ov, torch.bfloat16, "w_ov"), d_model, _ptr(o_lat, torch.float32, "o_lat"), M,
            _ptr(y, torch.float32, "y"), _stream(stream)))
        return y

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int32(0)
        self._check(self.lib.mla_get_device_status(self.h, _stream(stream), ctypes.byref(v)))
        return int(v.value)

    def debug_wait_timeout(self, limit_ns: int, stream=None):
        self._check(self.lib.mla_debug_wait_timeout(self.h, int(limit_ns), _stream(stream)))

    def decode_step(self, cache: Cache, w_uk, w_uv, q_nope, q_rope, q_pos, seq_lens,
                    scale: float = DEFAULT_SCALE, workspace=None, bufs=None, stream=None):
        """absorb_q -> decode_attn -> expand_v; returns (out, o_lat, lse)."""
        bufs = bufs or {}
        q_abs = self.absorb_q(w_uk, q_nope, q_rope, q_pos, bufs.get("q_abs"), stream)
        o_lat, lse = self.decode_attn(cache, q_abs, seq_lens, scale, workspace, bufs.get("o_lat"),
                                      bufs.get("lse"), stream)
        out = self.expand_v(w_uv, o_lat, bufs.get("out"), stream)
        return out, o_lat, lse


class DecodeStep:
    """One decode step for a fixed batch shape, over buffers it owns:

        append the new latent rows + absorb_q (one launch) -> decode_attn -> expand_v

    Write the step's inputs into ``c_kv, k_rope, seq_idx, pos`` (the new cache
    rows), ``q_nope, q_rope, q_pos`` and ``seq_lens``, then call ``run()``
    (direct launches on the current stream) or ``replay()`` (a CUDA graph made
    by ``capture()``; the graph keeps the buffer addresses, so refill the same
    tensors in place). Results: ``out`` [B,Hq,H,128] bf16, ``o_lat``, ``lse``.

    The eight input tensors are views into one device arena. ``host_inputs()``
    returns the same views of a pinned host arena; a graph captured with
    ``capture(host_io=True)`` copies that arena to the device with one copy kernel
    and runs the step with expand_v writing its result straight into the pinned
    ``out_host``, so one ``replay()`` plus a stream synchronize is a whole step
    from host memory to host memory.
    """

    _INPUTS = ("c_kv", "k_rope", "seq_idx", "pos", "q_nope", "q_rope", "q_pos", "seq_lens")

    def __init__(self, ctx: "Context", cache: Cache, w_uk, w_uv, B: int, Hq: int = 1,
                 scale: float = DEFAULT_SCALE, n_new=None, small: bool = False):
        """``small=True``: the step is one launch of mla_decode_step_small (short
        sequences, one new token per sequence: row b of c_kv / k_rope goes to
        position seq_lens[b] - 1; seq_idx, pos and q_pos are not read)."""
        torch = _torch()
        dev = w_uk.device
        H = int(w_uk.shape[0])
        self.ctx, self.cache, self.w_uk, self.w_uv = ctx, cache, w_uk, w_uv
        self.B, self.Hq, self.H, self.scale = B, Hq, H, scale
        self.small = bool(small)
        if self.small and (Hq != 1 or (n_new is not None and int(n_new) != B) or cache.fp8):
            raise ValueError("the one-launch step takes one new token per sequence (Hq = 1) over a bf16 cache")
        n = B * Hq if n_new is None else int(n_new)
        bf, i32 = torch.bfloat16, torch.int32
        self._layout = []           # (name, dtype, shape, byte offset) in the input arena
        off = 0
        for name, dt, shape in (("c_kv", bf, (n, D_C)), ("k_rope", bf, (n, D_ROPE)), ("seq_idx", i32, (n,)),
                                ("pos", i32, (n,)), ("q_nope", bf, (B, Hq, H, D_NOPE)),
                                ("q_rope", bf, (B, Hq, H, D_ROPE)), ("q_pos", i32, (B, Hq)), ("seq_lens", i32, (B,))):
            nbytes = int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
            self._layout.append((name, dt, shape, off, nbytes))
            off += (nbytes + 255) // 256 * 256
        self._arena = torch.zeros(max(off, 256), dtype=torch.uint8, device=dev)
        for name, t in self._views(self._arena).items():
            setattr(self, name, t)
        self.input_bytes = sum(e[4] for e in self._layout)
        self._host_arena = None
        self.out_host = None
        self.q_abs = torch.empty(B, Hq, H, ROW, dtype=bf, device=dev)
        self.o_lat = torch.empty(B, Hq, H, D_C, dtype=torch.float32, device=dev)
        self.lse = torch.empty(B, Hq, H, dtype=torch.float32, device=dev)
        self.out = torch.empty(B, Hq, H, D_V, dtype=bf, device=dev)
        self.workspace = None if self.small else ctx.alloc_workspace(H, B, Hq, dev)
        self.graph = None

    def _views(self, arena):
        return {name: arena[off:off + nbytes].view(dt).view(shape) for name, dt, shape, off, nbytes in self._layout}

    def host_inputs(self):
        """Pinned host views of the eight inputs (the arena ``capture(host_io=True)``
        copies to the device every replay); created on first use."""
        torch = _torch()
        if self._host_arena is None:
            self._host_arena = torch.zeros(self._arena.numel(), dtype=torch.uint8).pin_memory()
            self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        return self._views(self._host_arena)

    def run(self, stream=None, attn_events=None, out=None):
        """Launch the four calls; ``attn_events`` = (start, end) CUDA events
        recorded around the attention call; ``out``: where expand_v writes the
        result (default ``self.out``)."""
        c = self.ctx
        if self.small:
            if attn_events is not None:
                attn_events[0].record()
            c.decode_step_small(self.cache, self.c_kv, self.k_rope, self.w_uk, self.w_uv, self.q_nope, self.q_rope,
                                self.seq_lens, self.scale, self.out if out is None else out, self.o_lat, self.lse,
                                stream)
            if attn_events is not None:
                attn_events[1].record()
            return
        # append + absorb_q in one launch
        c.append_absorb_q(self.cache, self.c_kv, self.k_rope, self.seq_idx, self.pos, self.w_uk, self.q_nope,
                          self.q_rope, self.q_pos, self.q_abs, stream)
        if attn_events is not None:
            attn_events[0].record()
        c.decode_attn(self.cache, self.q_abs, self.seq_lens, self.scale, self.workspace, self.o_lat, self.lse,
                      stream)
        if attn_events is not None:
            attn_events[1].record()
        c.expand_v(self.w_uv, self.o_lat, self.out if out is None else out, stream)

    def capture(self, steps: int = 1, attn_events=None, host_io: bool = False):
        """Capture ``steps`` consecutive steps into one CUDA graph (after one
        direct warm-up step, which also prepares the kernels' attributes).
        ``attn_events``: optional list of ``steps`` (start, end) event pairs,
        created with ``external=True``, recorded inside the graph. ``host_io``:
        each step starts with the copy of the pinned host input arena
        (``host_inputs()``) to the device, and expand_v writes the result
        straight into the pinned ``out_host`` (the device addresses it directly)
        instead of ``out``."""
        torch = _torch()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        if host_io:
            self.host_inputs()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                if host_io:
                    self.ctx.copy_async(self._arena, self._host_arena)
                self.run(attn_events=None if attn_events is None else attn_events[i],
                         out=self.out_host if host_io else None)
        self.graph = g
        return g

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
