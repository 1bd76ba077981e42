"""ctypes binding of libfs_sample.so (the C ABI in include/fs_sample.h).

Argument marshalling only: tensors are passed as device pointers with the
current torch CUDA stream, and every step of the path runs in the library's
kernels.  torch is used for device memory and streams.  If the library is
missing, every call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfs_sample.so")

FS_OK = 0
FS_ERR_INVALID_ARG = 1
FS_ERR_UNSUPPORTED = 2
FS_ERR_CUDA = 3
FS_ERR_TIMEOUT = 4
FS_ERR_NO_MEMORY = 5
STATUS_NAMES = {0: "FS_OK", 1: "FS_ERR_INVALID_ARG", 2: "FS_ERR_UNSUPPORTED",
                3: "FS_ERR_CUDA", 4: "FS_ERR_TIMEOUT", 5: "FS_ERR_NO_MEMORY"}

FS_FLAG_NO_NOISE = 0x1
FS_FLAG_STORE_LOGITS = 0x2
FS_DTYPE_BF16 = 0
FS_DTYPE_F32 = 1
# Stage 1 launch forms (fs_stage1_form)
FS_STAGE1_ONE_CTA = 0
FS_STAGE1_MULTICAST_PAIR = 1
FS_STAGE1_PAIR_MMA = 2
STAGE1_FORM_NAMES = {FS_STAGE1_ONE_CTA: "one CTA per tile", FS_STAGE1_MULTICAST_PAIR: "multicast pair",
                     FS_STAGE1_PAIR_MMA: "pair MMA"}


class Transforms(ctypes.Structure):
    """fs_transforms of include/fs_sample.h."""
    _fields_ = [("bias", ctypes.c_void_p), ("softcap", ctypes.c_float),
                ("allow_mask", ctypes.c_void_p), ("mask_words", ctypes.c_int64)]


class FSError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


_lib = None

_i64, _u64, _u32, _f32, _int = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                ctypes.c_float, ctypes.c_int)
_vp, _sz = ctypes.c_void_p, ctypes.c_size_t

SIGNATURES = {
    "fs_sample": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _vp, _vp, _vp], _int),
    "fs_sample_host": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _vp, _vp, _vp],
                       _int),
    "fs_workspace_size": ([_i64, _i64, _i64], _sz),
    "fs_sample_ex": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _u32, _vp, _vp, _vp,
                      _vp, _sz, _vp], _int),
    "fs_stage1": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _u32, _vp, _vp, _sz, _vp],
                  _int),
    "fs_stage2": ([_i64, _i64, _i64, _f32, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "fs_sample_logprob": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _vp, _vp, _vp, _vp,
                           _sz, _vp], _int),
    "fs_sample_transformed": ([_vp, _vp, _i64, _i64, _i64, ctypes.c_void_p, _f32, _vp, _u64, _u64,
                               _u32, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "fs_sample_shard": ([_vp, _vp, _i64, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _vp, _vp, _vp,
                         _vp, _sz, _vp], _int),
    "fs_combine_groups": ([_i64, _i64, _vp, _vp, _u64, _u64, _vp, _vp, _vp], _int),
    "fs_logits_gemm": ([_vp, _vp, _i64, _i64, _i64, _vp, _int, _vp], _int),
    "fs_sample_from_logits": ([_vp, _int, _i64, _i64, _f32, _vp, _u64, _u64, _u32, _vp, _vp, _vp,
                               _sz, _vp], _int),
    "fs_sample_unfused": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _vp, _int, _vp, _vp,
                           _vp, _sz, _vp], _int),
    "fs_debug_noise": ([_u64, _u64, _i64, _i64, _i64, _vp, _vp, _vp], _int),
    "fs_debug_gumbel": ([_vp, _i64, _vp, _vp], _int),
    "fs_get_device_status": ([_vp, ctypes.POINTER(_u32)], _int),
    "fs_plan_info": ([_i64, _i64, _i64, _int, ctypes.POINTER(_i64)], _int),
    "fs_stage1_form": ([_i64, _i64, _i64, ctypes.POINTER(_int)], _int),
    "fs_release_workspaces": ([], _int),
    "fs_sample_noalloc": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _u64, _u64, _vp, _vp, _vp], _int),
    "fs_last_error_string": ([], ctypes.c_char_p),
    "fs_version": ([], ctypes.c_char_p),
}


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FSError(FS_ERR_UNSUPPORTED,
                          "libfs_sample.so is not built (run __graft_entry__.build() or "
                          "python exact_sampling_lm_gb300/build.py)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def _check(status: int):
    if status != FS_OK:
        raise FSError(status, lib().fs_last_error_string().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_matrix(name, t, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise FSError(FS_ERR_INVALID_ARG, "%s must be a CUDA tensor" % name)
    if t.dtype != dtype or t.dim() != 2 or not t.is_contiguous():
        raise FSError(FS_ERR_INVALID_ARG, "%s must be a contiguous 2-D %s tensor" % (name, dtype))


def _temps(temperature, device, B=None):
    """(scalar, per-row tensor or None) from a float or a [B] f32 CUDA tensor."""
    if isinstance(temperature, torch.Tensor):
        if temperature.dtype != torch.float32 or not temperature.is_cuda:
            raise FSError(FS_ERR_INVALID_ARG, "per-row temperatures must be f32 CUDA")
        if B is not None and temperature.numel() != B:
            raise FSError(FS_ERR_INVALID_ARG, "per-row temperatures must have B = %d entries, "
                          "got %d" % (B, temperature.numel()))
        return 1.0, temperature.contiguous()
    return float(temperature), None


# --------------------------------------------------------------------- entry points

def fs_version() -> str:
    return lib().fs_version().decode()


def fs_last_error_string() -> str:
    return lib().fs_last_error_string().decode()


def fs_plan_info(B: int, V: int, D: int, num_sms: int) -> dict:
    out = (_i64 * 6)()
    _check(lib().fs_plan_info(B, V, D, num_sms, out))
    keys = ("nM", "P", "G", "nCand", "ws_bytes", "max_tiles")
    return {k: int(v) for k, v in zip(keys, out)}


def fs_stage1_form(B: int, V: int, D: int) -> int:
    """The Stage 1 launch form (FS_STAGE1_*) for (B, V, D) on the current GPU."""
    out = _int(0)
    _check(lib().fs_stage1_form(B, V, D, ctypes.byref(out)))
    return int(out.value)


def fs_workspace_size(B: int, V: int, D: int) -> int:
    n = int(lib().fs_workspace_size(B, V, D))
    if n == 0:
        raise FSError(FS_ERR_INVALID_ARG, "fs_workspace_size failed: " + fs_last_error_string())
    return n


def workspace(B: int, V: int, D: int, device=None) -> torch.Tensor:
    """A caller workspace of fs_workspace_size bytes (uint8 CUDA tensor)."""
    n = fs_workspace_size(B, V, D)
    return torch.empty(n, dtype=torch.uint8, device=device or torch.cuda.current_device())


def _outs(B, device, out_idx, out_score, want_score):
    if out_idx is None:
        out_idx = torch.empty(B, dtype=torch.int64, device=device)
    if out_score is None and want_score:
        out_score = torch.empty(B, dtype=torch.float32, device=device)
    return out_idx, out_score


def fs_sample(H, W, temperature=1.0, seed=0, offset=0, out_idx=None, out_score=None,
              want_score=True, stream=None):
    """Sample one token per row of H from softmax(H W^T / T).  Returns (idx, score)."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    out_idx, out_score = _outs(B, H.device, out_idx, out_score, want_score)
    _check(lib().fs_sample(_ptr(H), _ptr(W), B, V, D, T, _ptr(Tv), seed, offset, _ptr(out_idx),
                           _ptr(out_score), _stream(stream)))
    return out_idx, out_score


def _check_host(name, t, dtype, dim):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise FSError(FS_ERR_INVALID_ARG, "%s must be a host (CPU) tensor" % name)
    if t.dtype != dtype or t.dim() != dim or not t.is_contiguous():
        raise FSError(FS_ERR_INVALID_ARG, "%s must be a contiguous %d-D %s tensor"
                      % (name, dim, dtype))


def fs_sample_host(H_host, W, temperature=1.0, seed=0, offset=0, out_idx=None, out_score=None,
                   want_score=True, stream=None):
    """fs_sample with H, per-row temperatures and the outputs in host memory (W on the
    device).  Outputs are valid once the stream reaches the end of the call; pinned
    buffers keep the copies asynchronous.  Returns (idx, score) host tensors."""
    _check_host("H_host", H_host, torch.bfloat16, 2)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H_host.shape
    V = W.shape[0]
    Tv = None
    if isinstance(temperature, torch.Tensor):
        _check_host("temperatures", temperature, torch.float32, 1)
        if temperature.numel() != B:
            raise FSError(FS_ERR_INVALID_ARG, "per-row temperatures must have B = %d entries, "
                          "got %d" % (B, temperature.numel()))
        T, Tv = 1.0, temperature
    else:
        T = float(temperature)
    if out_idx is None:
        out_idx = torch.empty(B, dtype=torch.int64).pin_memory()
    if out_score is None and want_score:
        out_score = torch.empty(B, dtype=torch.float32).pin_memory()
    _check_host("out_idx", out_idx, torch.int64, 1)
    if out_score is not None:
        _check_host("out_score", out_score, torch.float32, 1)
    if out_idx.numel() != B or (out_score is not None and out_score.numel() != B):
        raise FSError(FS_ERR_INVALID_ARG, "outputs must have B = %d entries" % B)
    _check(lib().fs_sample_host(_ptr(H_host), _ptr(W), B, V, D, T, _ptr(Tv), seed, offset,
                                _ptr(out_idx), _ptr(out_score), _stream(stream)))
    return out_idx, out_score


def fs_sample_ex(H, W, temperature=1.0, seed=0, offset=0, flags=0, out_idx=None,
                 out_score=None, out_logits=None, ws=None, want_score=True, stream=None):
    """fs_sample with flags / caller workspace.  Returns (idx, score, logits)."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    out_idx, out_score = _outs(B, H.device, out_idx, out_score, want_score)
    if (flags & FS_FLAG_STORE_LOGITS) and out_logits is None:
        out_logits = torch.empty((B, V), dtype=torch.float32, device=H.device)
    if ws is None:
        ws = workspace(B, V, D, H.device)
    _check(lib().fs_sample_ex(_ptr(H), _ptr(W), B, V, D, T, _ptr(Tv), seed, offset, flags,
                              _ptr(out_idx), _ptr(out_score), _ptr(out_logits), _ptr(ws),
                              ws.numel(), _stream(stream)))
    return out_idx, out_score, out_logits


def fs_sample_logprob(H, W, temperature=1.0, seed=0, offset=0, out_idx=None, out_score=None,
                      out_logprob=None, ws=None, want_score=True, stream=None):
    """fs_sample_ex plus the sampled token's log-probability.  Returns (idx, score, logprob)."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    out_idx, out_score = _outs(B, H.device, out_idx, out_score, want_score)
    if out_logprob is None:
        out_logprob = torch.empty(B, dtype=torch.float32, device=H.device)
    if ws is None:
        ws = workspace(B, V, D, H.device)
    _check(lib().fs_sample_logprob(_ptr(H), _ptr(W), B, V, D, T, _ptr(Tv), seed, offset,
                                   _ptr(out_idx), _ptr(out_score), _ptr(out_logprob), _ptr(ws),
                                   ws.numel(), _stream(stream)))
    return out_idx, out_score, out_logprob


def fs_sample_transformed(H, W, bias=None, softcap=0.0, allow_mask=None, temperature=1.0,
                          seed=0, offset=0, flags=0, want_logprob=False, out_idx=None,
                          out_score=None, ws=None, stream=None):
    """Fused sampling after bias [V] / soft-cap / allowed-token mask [B, words] (uint32 as
    int32).  Returns (idx, score, logprob or None)."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    out_idx, out_score = _outs(B, H.device, out_idx, out_score, True)
    lp = torch.empty(B, dtype=torch.float32, device=H.device) if want_logprob else None
    if ws is None:
        ws = workspace(B, V, D, H.device)
    tf = Transforms(_ptr(bias), float(softcap), _ptr(allow_mask),
                    0 if allow_mask is None else int(allow_mask.shape[1]))
    _check(lib().fs_sample_transformed(_ptr(H), _ptr(W), B, V, D, ctypes.addressof(tf), T,
                                       _ptr(Tv), seed, offset, flags, _ptr(out_idx),
                                       _ptr(out_score), _ptr(lp), _ptr(ws), ws.numel(),
                                       _stream(stream)))
    return out_idx, out_score, lp


def fs_sample_shard(H, W_shard, vocab_offset, temperature=1.0, seed=0, offset=0, ws=None,
                    stream=None):
    """Local sample (global index), score and log-mass of one vocabulary shard.
    Returns (idx int64 [B], score f32 [B], logmass f32 [B])."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W_shard", W_shard, torch.bfloat16)
    B, D = H.shape
    Vs = W_shard.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    idx = torch.empty(B, dtype=torch.int64, device=H.device)
    score = torch.empty(B, dtype=torch.float32, device=H.device)
    lm = torch.empty(B, dtype=torch.float32, device=H.device)
    if ws is None:
        ws = workspace(B, Vs, D, H.device)
    _check(lib().fs_sample_shard(_ptr(H), _ptr(W_shard), B, Vs, D, int(vocab_offset), T,
                                 _ptr(Tv), seed, offset, _ptr(idx), _ptr(score), _ptr(lm),
                                 _ptr(ws), ws.numel(), _stream(stream)))
    return idx, score, lm


def fs_combine_groups(group_idx, group_logmass, seed=0, offset=0, stream=None):
    """Grouped sampler over [G, B] local samples / log-masses.  Returns (idx, group)."""
    G, B = group_idx.shape
    gi = group_idx.contiguous()
    gl = group_logmass.contiguous()
    out = torch.empty(B, dtype=torch.int64, device=gi.device)
    grp = torch.empty(B, dtype=torch.int64, device=gi.device)
    _check(lib().fs_combine_groups(G, B, _ptr(gi), _ptr(gl), seed, offset, _ptr(out), _ptr(grp),
                                   _stream(stream)))
    return out, grp


def fs_stage1(H, W, ws, temperature=1.0, seed=0, offset=0, flags=0, out_logits=None,
              stream=None):
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    _check(lib().fs_stage1(_ptr(H), _ptr(W), B, V, D, T, _ptr(Tv), seed, offset, flags,
                           _ptr(out_logits), _ptr(ws), ws.numel(), _stream(stream)))


def fs_stage2(B, V, D, ws, temperature=1.0, out_idx=None, out_score=None, stream=None):
    T, Tv = _temps(temperature, ws.device, B)
    _check(lib().fs_stage2(B, V, D, T, _ptr(Tv), _ptr(out_idx), _ptr(out_score), _ptr(ws),
                           ws.numel(), _stream(stream)))
    return out_idx, out_score


def fs_logits_gemm(H, W, Y=None, y_dtype=FS_DTYPE_BF16, stream=None):
    """Unfused GEMM: returns Y = H W^T as bf16 or f32 [B, V]."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    if Y is None:
        dt = torch.float32 if y_dtype == FS_DTYPE_F32 else torch.bfloat16
        Y = torch.empty((B, V), dtype=dt, device=H.device)
    _check(lib().fs_logits_gemm(_ptr(H), _ptr(W), B, V, D, _ptr(Y), y_dtype, _stream(stream)))
    return Y


def fs_sample_from_logits(Y, temperature=1.0, seed=0, offset=0, flags=0, out_idx=None,
                          out_score=None, ws=None, want_score=True, stream=None):
    """Gumbel-max over materialised logits Y [B, V] (bf16 or f32)."""
    if Y.dtype == torch.float32:
        y_dtype = FS_DTYPE_F32
    elif Y.dtype == torch.bfloat16:
        y_dtype = FS_DTYPE_BF16
    else:
        raise FSError(FS_ERR_INVALID_ARG, "Y must be bf16 or f32")
    if not Y.is_cuda or Y.dim() != 2 or not Y.is_contiguous():
        raise FSError(FS_ERR_INVALID_ARG, "Y must be a contiguous 2-D CUDA tensor")
    B, V = Y.shape
    T, Tv = _temps(temperature, Y.device, Y.shape[0])
    out_idx, out_score = _outs(B, Y.device, out_idx, out_score, want_score)
    if ws is None:
        ws = workspace(B, V, 8, Y.device)
    _check(lib().fs_sample_from_logits(_ptr(Y), y_dtype, B, V, T, _ptr(Tv), seed, offset, flags,
                                       _ptr(out_idx), _ptr(out_score), _ptr(ws), ws.numel(),
                                       _stream(stream)))
    return out_idx, out_score


def fs_sample_unfused(H, W, temperature=1.0, seed=0, offset=0, Y=None, y_dtype=FS_DTYPE_BF16,
                      out_idx=None, out_score=None, ws=None, want_score=True, stream=None):
    """The unfused comparator: GEMM writing Y, then a sampling pass over Y."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    out_idx, out_score = _outs(B, H.device, out_idx, out_score, want_score)
    if Y is None:
        dt = torch.float32 if y_dtype == FS_DTYPE_F32 else torch.bfloat16
        Y = torch.empty((B, V), dtype=dt, device=H.device)
    if ws is None:
        ws = workspace(B, V, D, H.device)
    _check(lib().fs_sample_unfused(_ptr(H), _ptr(W), B, V, D, T, _ptr(Tv), seed, offset,
                                   _ptr(Y), y_dtype, _ptr(out_idx), _ptr(out_score), _ptr(ws),
                                   ws.numel(), _stream(stream)))
    return out_idx, out_score, Y


def fs_debug_noise(seed, offset, b0, nb, V, device=None, stream=None):
    """(words uint32-as-int32 [nb, V], g f32 [nb, V]) from the device noise functions."""
    dev = device or torch.cuda.current_device()
    words = torch.empty((nb, V), dtype=torch.int32, device=dev)
    g = torch.empty((nb, V), dtype=torch.float32, device=dev)
    _check(lib().fs_debug_noise(seed, offset, b0, nb, V, _ptr(words), _ptr(g), _stream(stream)))
    return words, g


def fs_debug_gumbel(words, stream=None):
    """g f32 [n] of the device Gumbel transform applied to uint32 words (as int32) [n]."""
    if not isinstance(words, torch.Tensor) or not words.is_cuda or words.dtype != torch.int32 \
            or not words.is_contiguous():
        raise FSError(FS_ERR_INVALID_ARG, "words must be a contiguous int32 CUDA tensor")
    g = torch.empty(words.shape, dtype=torch.float32, device=words.device)
    _check(lib().fs_debug_gumbel(_ptr(words), words.numel(), _ptr(g), _stream(stream)))
    return g


def fs_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    w = _u32(0)
    st = lib().fs_get_device_status(_stream(stream), ctypes.byref(w))
    if st not in (FS_OK, FS_ERR_TIMEOUT):
        _check(st)
    return int(w.value)


def fs_sample_noalloc(H, W, temperature=1.0, seed=0, offset=0, out_idx=None, out_score=None,
                      want_score=True, stream=None):
    """fs_sample without any device allocation by the library (static scratch).
    Output tensors are allocated here by torch unless the caller passes them."""
    _check_matrix("H", H, torch.bfloat16)
    _check_matrix("W", W, torch.bfloat16)
    B, D = H.shape
    V = W.shape[0]
    T, Tv = _temps(temperature, H.device, H.shape[0])
    out_idx, out_score = _outs(B, H.device, out_idx, out_score, want_score)
    _check(lib().fs_sample_noalloc(_ptr(H), _ptr(W), B, V, D, T, _ptr(Tv), seed, offset,
                                   _ptr(out_idx), _ptr(out_score), _stream(stream)))
    return out_idx, out_score


def fs_release_workspaces():
    _check(lib().fs_release_workspaces())
