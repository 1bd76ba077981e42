"""Host-side checks of the C ABI (no GPU needed).

The shared library must load, export every function include/fs_sample.h
declares, describe its schedule, and reject bad arguments with a status and a
message before touching the GPU.
"""
import ctypes
import os
import re

import pytest
import torch

import exact_sampling_lm_gb300 as fs
from exact_sampling_lm_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_sampling_lm_gb300 import build
    build.build()


def declared_functions():
    names = []
    for fname in sorted(os.listdir(HEADER_DIR)):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(fs_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("fs_sample", "fs_sample_ex", "fs_stage1", "fs_stage2", "fs_workspace_size",
                 "fs_logits_gemm", "fs_sample_from_logits", "fs_sample_unfused",
                 "fs_debug_noise", "fs_get_device_status", "fs_last_error_string",
                 "fs_version", "fs_plan_info", "fs_stage1_form", "fs_release_workspaces"):
        assert must in names


def test_library_exports_every_declared_symbol():
    handle = ctypes.CDLL(_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(handle, name), name
        assert name in _lib.SIGNATURES, "binding lacks " + name


def test_version_and_error_string():
    assert "sm_103a" in fs.fs_version()
    assert isinstance(fs.fs_last_error_string(), str)


@pytest.mark.parametrize("B,V,D,sms", [(1, 128256, 4096, 152), (64, 128256, 4096, 152),
                                       (256, 151936, 3584, 152), (1024, 128256, 8192, 152),
                                       (512, 262144, 2304, 152), (4, 4096, 256, 152),
                                       (300, 50257, 72, 148), (3, 5, 8, 152)])
def test_plan_covers_the_vocabulary(B, V, D, sms):
    """Partitions are disjoint, cover [0, V) in 16-row units, and every CTA
    gets at most max_tiles tiles (balanced tiles of <= 256 rows, then a final
    128-row tile); one CTA per SM at most."""
    p = fs.fs_plan_info(B, V, D, sms)
    nM = (B + 127) // 128
    assert p["nM"] == nM
    assert p["G"] == p["P"] * nM <= max(sms, nM)
    assert p["nCand"] == p["P"]
    U = (V + 15) // 16
    covered = 0
    for part in range(p["P"]):
        u0 = part * U // p["P"]
        u1 = (part + 1) * U // p["P"]
        r0, r1 = 16 * u0, min(16 * u1, V)
        assert r0 == covered
        covered = r1
        nu = u1 - u0
        if nM % 2 == 0:  # paired CTAs: plain 256-row tiles
            tiles = (r1 - r0 + 255) // 256
        else:
            tiles = 1 if nu <= 16 else (nu - 8 + 15) // 16 + 1
        assert tiles <= p["max_tiles"]
        assert r1 > r0
    assert covered == V
    slots = max(p["nCand"], logits_sampler_chunks(B, V, sms))
    assert p["ws_bytes"] == 5 * ((slots * B * 4 + 255) // 256 * 256)


def logits_sampler_chunks(B, V, sms):
    """Blocks per row of the materialised-logits sampler: chunks of 2 K .. 64 K
    entries (multiples of 2048), sized for about 4 blocks per SM over B x V."""
    step = 2048
    chunk = -(-(B * V // (4 * sms)) // step) * step
    chunk = max(step, min(chunk, 65536, -(-V // step) * step))
    return -(-V // chunk)


def call_sample(H=16, W=16, B=4, V=64, D=64, T=1.0, temps=None, out=16):
    return _lib.lib().fs_sample(H, W, B, V, D, T, temps, 0, 0, out, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(H=None), _lib.FS_ERR_INVALID_ARG),
    (dict(W=None), _lib.FS_ERR_INVALID_ARG),
    (dict(out=None), _lib.FS_ERR_INVALID_ARG),
    (dict(B=0), _lib.FS_ERR_INVALID_ARG),
    (dict(V=0), _lib.FS_ERR_INVALID_ARG),
    (dict(D=0), _lib.FS_ERR_INVALID_ARG),
    (dict(D=12), _lib.FS_ERR_UNSUPPORTED),
    (dict(H=24), _lib.FS_ERR_UNSUPPORTED),
    (dict(W=8), _lib.FS_ERR_UNSUPPORTED),
    (dict(V=2**31), _lib.FS_ERR_UNSUPPORTED),
    (dict(B=2**24 + 1), _lib.FS_ERR_UNSUPPORTED),
    (dict(T=0.0), _lib.FS_ERR_INVALID_ARG),
    (dict(T=-1.0), _lib.FS_ERR_INVALID_ARG),
    (dict(T=float("inf")), _lib.FS_ERR_INVALID_ARG),
    (dict(T=float("nan")), _lib.FS_ERR_INVALID_ARG),
])
def test_bad_arguments_are_rejected_before_any_launch(kw, status):
    assert call_sample(**kw) == status
    assert len(fs.fs_last_error_string()) > 0


def test_other_entry_points_validate():
    L = _lib.lib()
    assert L.fs_stage1(16, 16, 4, 64, 64, 1.0, None, 0, 0, 0x80, None, 16, 1 << 20, None) \
        == _lib.FS_ERR_INVALID_ARG  # unknown flag
    assert L.fs_stage1(16, 16, 4, 64, 64, 1.0, None, 0, 0, _lib.FS_FLAG_STORE_LOGITS, None, 16,
                       1 << 20, None) == _lib.FS_ERR_INVALID_ARG  # logits buffer missing
    assert L.fs_logits_gemm(16, 16, 4, 64, 64, 16, 7, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_sample_from_logits(16, 0, 4, 64, 1.0, None, 0, 0, _lib.FS_FLAG_STORE_LOGITS,
                                   16, None, 16, 1 << 20, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_debug_noise(0, 0, -1, 1, 8, 16, None, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_debug_noise(0, 0, 0, 1, 8, None, None, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_debug_gumbel(None, 8, 16, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_debug_gumbel(16, 0, 16, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_debug_gumbel(18, 8, 16, None) == _lib.FS_ERR_UNSUPPORTED
    out = (ctypes.c_int64 * 6)()
    assert L.fs_plan_info(4, 64, 64, 0, out) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_workspace_size(0, 64, 64) == 0


def test_shard_and_combine_entries_validate():
    """Vocabulary shards: the offset is a non-negative multiple of 16 and the
    shard's last global index stays below 2^31 - 1; the grouped combine needs
    at least one group and at most 2^24 rows.  All refused before any launch."""
    L = _lib.lib()

    def shard(vocab_offset, V=64, logmass=48):
        return L.fs_sample_shard(16, 32, 4, V, 64, vocab_offset, 1.0, None, 0, 0, 16, None,
                                 logmass, 64, 1 << 20, None)

    assert shard(8) == _lib.FS_ERR_INVALID_ARG
    assert shard(-16) == _lib.FS_ERR_INVALID_ARG
    # offset + V = 2^31: the last global index would be 2^31 - 1 (every case
    # here is refused by validation, so no call reaches a device)
    assert shard(2**31 - 64, V=64) == _lib.FS_ERR_UNSUPPORTED
    assert shard(2**31 - 80, V=80) == _lib.FS_ERR_UNSUPPORTED
    assert shard(0, logmass=None) == _lib.FS_ERR_INVALID_ARG
    assert shard(0, logmass=50) == _lib.FS_ERR_UNSUPPORTED         # misaligned log-mass output
    assert L.fs_combine_groups(0, 4, 16, 32, 0, 0, 48, 64, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_combine_groups(2, 2**24 + 1, 16, 32, 0, 0, 48, 64, None) == _lib.FS_ERR_UNSUPPORTED
    assert L.fs_combine_groups(2, 4, None, 32, 0, 0, 48, 64, None) == _lib.FS_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_call_without_a_device_reports_cuda_error():
    """With valid arguments but no GPU the call fails with FS_ERR_CUDA (or
    UNSUPPORTED) instead of crashing: there is no CPU fallback."""
    st = call_sample()
    assert st in (_lib.FS_ERR_CUDA, _lib.FS_ERR_UNSUPPORTED)


def test_stage1_form_validates_before_touching_a_device():
    L = _lib.lib()
    out = ctypes.c_int(-1)
    assert L.fs_stage1_form(256, 4096, 64, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_stage1_form(0, 4096, 64, ctypes.byref(out)) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_stage1_form(256, 4096, 60, ctypes.byref(out)) == _lib.FS_ERR_UNSUPPORTED  # D % 8
    assert out.value == -1


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_stage1_form_without_a_device_reports_an_error():
    out = ctypes.c_int(-1)
    st = _lib.lib().fs_stage1_form(256, 4096, 64, ctypes.byref(out))
    assert st in (_lib.FS_ERR_CUDA, _lib.FS_ERR_UNSUPPORTED) and out.value == -1


def test_transformed_entry_validates():
    L = _lib.lib()
    ws = 1 << 20
    tf = _lib.Transforms(None, -1.0, None, 0)
    assert L.fs_sample_transformed(16, 16, 4, 64, 64, ctypes.addressof(tf), 1.0, None, 0, 0, 0,
                                   16, None, None, 16, ws, None) == _lib.FS_ERR_INVALID_ARG
    tf = _lib.Transforms(8, 0.0, None, 0)  # misaligned bias
    assert L.fs_sample_transformed(16, 16, 4, 64, 64, ctypes.addressof(tf), 1.0, None, 0, 0, 0,
                                   16, None, None, 16, ws, None) == _lib.FS_ERR_UNSUPPORTED
    tf = _lib.Transforms(None, 0.0, 16, 1)  # V=64 needs 2 mask words
    assert L.fs_sample_transformed(16, 16, 4, 64, 64, ctypes.addressof(tf), 1.0, None, 0, 0, 0,
                                   16, None, None, 16, ws, None) == _lib.FS_ERR_INVALID_ARG
    assert L.fs_sample_transformed(16, 16, 4, 64, 64, None, 1.0, None, 0, 0, 0,
                                   16, None, None, 16, ws, None) == _lib.FS_ERR_INVALID_ARG
    tf = _lib.Transforms(None, 0.0, None, 0)
    assert L.fs_sample_transformed(16, 16, 4, 64, 64, ctypes.addressof(tf), 1.0, None, 0, 0, 2,
                                   16, None, None, 16, ws, None) == _lib.FS_ERR_INVALID_ARG


def test_misaligned_outputs_are_rejected():
    L = _lib.lib()
    # out_idx must be 8-byte aligned, out_score 4-byte aligned
    assert L.fs_sample(16, 16, 4, 64, 64, 1.0, None, 0, 0, 20, None, None) == \
        _lib.FS_ERR_UNSUPPORTED
    assert L.fs_sample(16, 16, 4, 64, 64, 1.0, None, 0, 0, 16, 18, None) == \
        _lib.FS_ERR_UNSUPPORTED
    assert L.fs_sample(16, 16, 4, 64, 64, 1.0, 6, 0, 0, 16, None, None) == \
        _lib.FS_ERR_UNSUPPORTED


def test_sample_ex_checks_outputs_before_stage1():
    """fs_sample_ex checks Stage 2's outputs before Stage 1 launches: a
    misaligned out_score or out_idx is refused before any device call (on a
    machine without a GPU the status is the validation error, not a CUDA
    error from the device query)."""
    L = _lib.lib()
    ws = 1 << 20
    assert L.fs_sample_ex(16, 16, 4, 64, 64, 1.0, None, 0, 0, 0, 16, 18, None, 32, ws, None) == \
        _lib.FS_ERR_UNSUPPORTED
    assert L.fs_sample_ex(16, 16, 4, 64, 64, 1.0, None, 0, 0, 0, 20, None, None, 32, ws, None) == \
        _lib.FS_ERR_UNSUPPORTED
    assert "aligned" in fs.fs_last_error_string()


def test_binding_checks_per_row_temperature_length():
    from exact_sampling_lm_gb300 import _lib as b
    with pytest.raises(b.FSError):
        b._temps(torch.ones(3), "cpu", 4)  # not CUDA


def test_host_buffer_entry_validates():
    L = _lib.lib()
    # H_host, W and out_idx_host are required; host pointers need no alignment
    assert L.fs_sample_host(None, 16, 4, 64, 64, 1.0, None, 0, 0, 16, None, None) == \
        _lib.FS_ERR_INVALID_ARG
    assert L.fs_sample_host(16, None, 4, 64, 64, 1.0, None, 0, 0, 16, None, None) == \
        _lib.FS_ERR_INVALID_ARG
    assert L.fs_sample_host(16, 16, 4, 64, 64, 1.0, None, 0, 0, None, None, None) == \
        _lib.FS_ERR_INVALID_ARG
    assert L.fs_sample_host(16, 8, 4, 64, 64, 1.0, None, 0, 0, 16, None, None) == \
        _lib.FS_ERR_UNSUPPORTED  # W is the device operand of the TMA loads
    assert L.fs_sample_host(16, 16, 4, 64, 12, 1.0, None, 0, 0, 16, None, None) == \
        _lib.FS_ERR_UNSUPPORTED
    assert L.fs_sample_host(16, 16, 0, 64, 64, 1.0, None, 0, 0, 16, None, None) == \
        _lib.FS_ERR_INVALID_ARG
    assert L.fs_sample_host(16, 16, 4, 64, 64, 0.0, None, 0, 0, 16, None, None) == \
        _lib.FS_ERR_INVALID_ARG


def test_host_buffer_binding_rejects_device_or_wrong_tensors():
    W = torch.zeros(64, 64, dtype=torch.bfloat16)
    H = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(fs.FSError):  # W must be a CUDA tensor
        fs.fs_sample_host(H, W)
    with pytest.raises(fs.FSError):  # H must be bf16
        fs.fs_sample_host(H.float(), W)
    with pytest.raises(fs.FSError):  # H must be contiguous
        fs.fs_sample_host(torch.zeros(64, 4, dtype=torch.bfloat16).t(), W)
