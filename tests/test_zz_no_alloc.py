"""fs_sample_noalloc: fs_sample for callers that cannot allocate device memory.

Some callers own every byte of device memory themselves: an inference server
that reserves its pool at start-up and forbids allocation afterwards, a
plug-in whose host process controls the allocator.  Others sit on a
latency-critical decode step where cudaMalloc, which may synchronise the
device, is not acceptable.  fs_sample_noalloc serves them: its candidate
scratch is a static array inside the library, so it allocates nothing.

These tests call it through the C ABI and compare it with fs_sample (the
allocating entry point) on two calls in a row, where the second call reuses
the scratch the first one left behind; indices and scores must agree exactly,
the bar the parity tests use for indices.  An oversized request must be
refused before anything is launched.  This file is collected last so that a
failure here never hides the other tests.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 1 << 20  # FS_NOALLOC_SCRATCH_BYTES in include/fs_sample.h


@pytest.fixture(scope="module")
def fs():
    import exact_sampling_lm_gb300 as fs_mod
    from exact_sampling_lm_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    return fs_mod


def noalloc_call(fs, H, W, T, seed, offset):
    """fs_sample_noalloc through the C ABI with raw device pointers."""
    B, D = H.shape
    V = W.shape[0]
    idx = torch.empty(B, dtype=torch.int64, device=H.device)
    score = torch.empty(B, dtype=torch.float32, device=H.device)
    per_row = isinstance(T, torch.Tensor)
    st = fs.lib().fs_sample_noalloc(
        H.data_ptr(), W.data_ptr(), B, V, D, 1.0 if per_row else float(T),
        T.data_ptr() if per_row else None, seed, offset, idx.data_ptr(), score.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, fs.fs_last_error_string()
    return idx, score


@pytest.mark.parametrize("B,V,D,T", [(64, 50000, 256, 1.0), (300, 20011, 64, "rows"),
                                     (256, 30011, 192, 0.7), (1, 4099, 136, 1.3)])
def test_noalloc_matches_fs_sample_on_two_calls(fs, B, V, D, T):
    g = torch.Generator(device="cpu").manual_seed(B * 31 + V)
    dev = torch.device("cuda:0")
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    if T == "rows":
        T = (0.5 + torch.rand(B, generator=g)).to(dev)
    for offset in (11, 12):
        a_idx, a_score = noalloc_call(fs, H, W, T, 4242, offset)
        b_idx, b_score = fs.fs_sample(H, W, temperature=T, seed=4242, offset=offset)
        torch.cuda.synchronize()
        assert torch.equal(a_idx, b_idx)
        assert torch.equal(a_score, b_score)
    assert fs.fs_get_device_status() == 0


def sample_scratch_bytes(B, V):
    """The two candidate arrays (score, index) plain sampling keeps: each
    P x B four-byte values rounded to 256 B, P being Stage 1's vocabulary
    partitions, min(SMs // ceil(B / 128), ceil(V / 16)), at least 1."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    parts = max(1, min(sms // ((B + 127) // 128), (V + 15) // 16))
    return 2 * ((parts * B * 4 + 255) // 256 * 256)


def test_noalloc_takes_what_only_the_two_sampling_arrays_fit(fs):
    """A shape whose full workspace (five arrays wide enough for every entry
    point) exceeds the scratch while the two arrays that sampling keeps fit:
    the call is accepted and agrees with fs_sample."""
    B, D = 32768, 64
    V = next(v for v in (4096, 16384, 65536, 262144)
             if fs.fs_workspace_size(B, v, D) > SCRATCH_BYTES >= sample_scratch_bytes(B, v))
    g = torch.Generator(device="cpu").manual_seed(77)
    dev = torch.device("cuda:0")
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    for offset in (3, 4):
        a_idx, a_score = noalloc_call(fs, H, W, 0.9, 99, offset)
        b_idx, b_score = fs.fs_sample(H, W, temperature=0.9, seed=99, offset=offset)
        torch.cuda.synchronize()
        assert torch.equal(a_idx, b_idx) and torch.equal(a_score, b_score)


def test_noalloc_refuses_requests_beyond_its_scratch(fs):
    B, V, D = 262144, 16, 8
    assert sample_scratch_bytes(B, V) > SCRATCH_BYTES
    dev = torch.device("cuda:0")
    H = torch.zeros((B, D), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((V, D), dtype=torch.bfloat16, device=dev)
    idx = torch.full((B,), -7, dtype=torch.int64, device=dev)
    st = fs.lib().fs_sample_noalloc(H.data_ptr(), W.data_ptr(), B, V, D, 1.0, None, 0, 0,
                                    idx.data_ptr(), None, None)
    assert st == 2  # FS_ERR_UNSUPPORTED
    assert "scratch" in fs.fs_last_error_string()
    torch.cuda.synchronize()
    assert torch.all(idx == -7)  # nothing was launched
