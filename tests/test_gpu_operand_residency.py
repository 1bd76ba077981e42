"""Stage 1 reads H and W only from the calling GPU's own memory.

Its TMA tensor maps are encoded on the caller's pointers, and in the paired
forms both CTAs of a cluster share W boxes (multicast) or feed one MMA.  The entry points
check where H and W live before encoding anything: page-locked host memory
(reachable through a mapping) and pageable host memory are refused with
FS_ERR_UNSUPPORTED, nothing is launched, and the outputs stay untouched.
Every call here is refused on the host, so no kernel runs.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

FS_ERR_UNSUPPORTED = 2


@pytest.fixture(scope="module")
def fs():
    import exact_sampling_lm_gb300 as fs_mod
    from exact_sampling_lm_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    return fs_mod


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("where", ["pinned", "pageable"])
@pytest.mark.parametrize("operand", ["W", "H"])
def test_host_operands_are_refused(fs, where, operand):
    B, V, D = 256, 4096, 64  # B = 256: a paired shape
    dev = torch.device("cuda:0")
    H = torch.zeros((B, D), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((V, D), dtype=torch.bfloat16, device=dev)
    host = torch.zeros(((V if operand == "W" else B), D), dtype=torch.bfloat16,
                       pin_memory=(where == "pinned"))
    if operand == "W":
        W = host
    else:
        H = host
    idx = torch.full((B,), -7, dtype=torch.int64, device=dev)
    score = torch.full((B,), 3.0, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    L = fs.lib()
    st = L.fs_sample(H.data_ptr(), W.data_ptr(), B, V, D, 1.0, None, 1, 2, idx.data_ptr(),
                     score.data_ptr(), _stream())
    assert st == FS_ERR_UNSUPPORTED
    msg = fs.fs_last_error_string()
    assert operand in msg and "device memory of the current GPU" in msg, msg
    ws = fs.workspace(B, V, D)
    st = L.fs_sample_ex(H.data_ptr(), W.data_ptr(), B, V, D, 1.0, None, 1, 2, 0, idx.data_ptr(),
                        score.data_ptr(), None, ws.data_ptr(), ws.numel(), _stream())
    assert st == FS_ERR_UNSUPPORTED
    y = torch.full((B, V), 5.0, dtype=torch.float32, device=dev)
    st = L.fs_logits_gemm(H.data_ptr(), W.data_ptr(), B, V, D, y.data_ptr(), 1, _stream())
    assert st == FS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(idx == -7) and torch.all(score == 3.0) and torch.all(y == 5.0)
    assert fs.fs_get_device_status() == 0


def test_host_buffer_call_refuses_a_host_W_before_its_upload(fs):
    """fs_sample_host takes H from the host by design, but W must be device
    memory; the refusal comes before the upload kernel launches."""
    B, V, D = 8, 4096, 64
    H = torch.ones((B, D), dtype=torch.bfloat16).pin_memory()
    W = torch.zeros((V, D), dtype=torch.bfloat16).pin_memory()
    idx = torch.full((B,), -7, dtype=torch.int64).pin_memory()
    st = fs.lib().fs_sample_host(H.data_ptr(), W.data_ptr(), B, V, D, 1.0, None, 1, 2,
                                 idx.data_ptr(), None, _stream())
    assert st == FS_ERR_UNSUPPORTED
    assert "W" in fs.fs_last_error_string()
    torch.cuda.synchronize()
    assert torch.all(idx == -7)


def test_device_operands_still_accepted(fs):
    B, V, D = 256, 4096, 64
    dev = torch.device("cuda:0")
    g = torch.Generator(device="cpu").manual_seed(5)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    i1, s1 = fs.fs_sample(H, W, temperature=1.0, seed=1, offset=2)
    i2, s2, _ = fs.fs_sample_ex(H, W, temperature=1.0, seed=1, offset=2)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(s1, s2)
    assert bool(torch.all((i1 >= 0) & (i1 < V)))
