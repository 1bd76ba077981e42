"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars (FlashSampling's exactness claim: the tiled kernel returns the same
maximizer as a full Gumbel-max pass, Appendix C):
  * noise words bit-exact; Gumbels within 4 ulp(g) + 1e-6 of the oracle's
    double-precision value rounded to f32;
  * logits within |dl| <= 2e-2 of the oracle's logits (bf16 inputs, f32
    accumulation: the oracle sums in index order, the tensor cores in their
    own order);
  * sampled indices bit-exact, except where the oracle's two best perturbed
    scores are closer than 1e-3 (a near-tie, where the f32 rounding of a
    different summation order may decide); near-ties are counted and printed.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-2
NEAR_TIE = 1e-3


@pytest.fixture(scope="module")
def fs():
    import exact_sampling_lm_gb300 as fs_mod
    from exact_sampling_lm_gb300 import build
    build.build()
    return fs_mod


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def bits(t):
    return workloads.to_bits(t)


def host_T(T, B):
    if isinstance(T, torch.Tensor):
        return T.detach().cpu().numpy().astype(np.float32)
    return np.full(B, T, dtype=np.float32)


def compare_indices(g_idx, o_idx, o_best, o_second, label=""):
    near = (o_best - o_second) < NEAR_TIE
    mism = g_idx != o_idx
    bad = mism & ~near
    assert not bad.any(), "%s: %d index mismatches away from near-ties at rows %s" % (
        label, int(bad.sum()), np.nonzero(bad)[0][:10])
    n_near_mism = int((mism & near).sum())
    print("[%s] rows=%d near-ties=%d near-tie mismatches=%d" % (label, len(g_idx),
                                                               int(near.sum()), n_near_mism))
    return n_near_mism


def run_and_check(fs, H, W, T, seed, offset, label, flags=0, store=True, rows=None):
    """Fused path vs oracle.  rows: subset of rows to check (None = all)."""
    B, D = H.shape
    V = W.shape[0]
    f = flags | (fs.FS_FLAG_STORE_LOGITS if store else 0)
    idx, score, logits = fs.fs_sample_ex(H, W, temperature=T, seed=seed, offset=offset, flags=f)
    torch.cuda.synchronize()
    assert fs.fs_get_device_status() == 0
    rows = np.arange(B) if rows is None else np.asarray(rows)
    Hb = bits(H)[rows]
    Wb = bits(W)
    Th = host_T(T, B)[rows]
    o_idx, o_best, o_second, o_l32 = oracle.sample(Hb, Wb, Th, seed, offset,
                                                   flags=(oracle.NO_NOISE if flags & 1 else 0),
                                                   want_logits=store, row_ids=rows)
    g_idx = idx.cpu().numpy()[rows]
    if store:
        gl = logits[torch.as_tensor(rows, device=logits.device)].cpu().numpy().astype(np.float64)
        dl = np.abs(gl - o_l32.astype(np.float64)).max()
        assert dl <= LOGIT_TOL, "%s: max |dl| = %g" % (label, dl)
        print("[%s] max |dl| = %.3e" % (label, dl))
    compare_indices(g_idx, o_idx, o_best, o_second, label)
    g_score = score.cpu().numpy()[rows]
    same = g_idx == o_idx
    valid = same & np.isfinite(o_best)
    if valid.any():
        ds = np.abs(g_score[valid] - o_best[valid])
        lim = LOGIT_TOL / np.minimum(Th[valid], 1.0) + 1e-5
        assert np.all(ds <= lim), "%s: winning score differs by %g" % (label, ds.max())
    invalid = ~(np.isfinite(Th) & (Th > 0))
    assert np.all(g_idx[invalid] == -1) and np.all(np.isnan(g_score[invalid]))
    return idx, score


# ---------------------------------------------------------------- noise

def test_noise_words_bit_exact_and_gumbel_within_bound(fs, dev):
    for seed, offset, b0, nb, V in [(0x5EED0040, 0, 0, 256, 4099), (2**64 - 1, 2**63, 17, 64, 8192),
                                    (12345, 7, 1 << 20, 1024, 16384)]:
        words, g = fs.fs_debug_noise(seed, offset, b0, nb, V)
        torch.cuda.synchronize()
        o_words, o_g = oracle.noise_block(seed, offset, b0, nb, 0, V)
        assert np.array_equal(words.cpu().numpy().view(np.uint32), o_words)
        gg = g.cpu().numpy().astype(np.float64)
        og = o_g.astype(np.float64)
        ulp = np.spacing(np.abs(o_g)).astype(np.float64)
        err = np.abs(gg - og)
        assert np.all(err <= 4 * ulp + 1e-6), "max err %g" % err.max()
        print("noise block %dx%d: max |dg| = %.3e, max in ulps = %.2f" % (
            nb, V, err.max(), float((err / ulp).max())))


def test_gumbel_transform_exhaustive(fs, dev):
    """Every one of the 2^23 distinct uniforms u = k 2^-24 (k odd): the device
    Gumbel is within 2 ulp(g) + 3e-7 of the oracle's (double, rounded once).
    That bound covers w = -log u to about 1 ulp and the hardware log2's
    absolute error of about 2^-22 in the outer logarithm."""
    k = np.arange(1, 1 << 24, 2, dtype=np.uint32)
    words = (k << np.uint32(8)).view(np.int32)
    g = fs.fs_debug_gumbel(torch.from_numpy(words).to(dev))
    torch.cuda.synchronize()
    gg = g.cpu().numpy().astype(np.float64)
    og = oracle.gumbel_block(words.view(np.uint32)).astype(np.float64)
    ulp = np.spacing(np.abs(og).astype(np.float32)).astype(np.float64)
    err = np.abs(gg - og)
    bad = err > 2 * ulp + 3e-7
    assert not bad.any(), "%d uniforms out of bound, first k = %d (err %g)" % (
        int(bad.sum()), int(k[bad][0]), float(err[bad][0]))
    # the series branch (u >= 15/16) holds the large Gumbels that win
    hi = k >= (15 << 20)
    print("gumbel: max |dg| = %.3e overall, %.3e for u >= 15/16; max in ulps %.2f" % (
        err.max(), err[hi].max(), float((err / ulp).max())))


# ---------------------------------------------------------------- small exhaustive cases

def test_tiny_workload(fs, dev):
    B = 4
    H = workloads.make_hidden("tiny", B).to(dev)
    W = workloads.make_weights("tiny").to(dev)
    seed, offset = workloads.sampling_seed("tiny", B)
    for off in (offset, offset + 1, offset + 12345):
        run_and_check(fs, H, W, 1.0, seed, off, "tiny off=%d" % off)


@pytest.mark.parametrize("B,V,D", [
    (1, 5, 8), (3, 17, 16), (5, 100, 72), (1, 4096, 256), (7, 4099, 136),
    (127, 2000, 64), (128, 2048, 128), (129, 3001, 64), (255, 1000, 520),
    (300, 5003, 200), (2, 50257, 64), (33, 40000, 64), (130, 41000, 96),
    (16, 45000, 136), (17, 45000, 136), (88, 45000, 200), (89, 45000, 200),
    (96, 45000, 64), (97, 45000, 64), (256, 1000, 8192), (256, 64, 65536),
    (256, 3001, 4032), (256, 3001, 4096), (512, 1000, 6080), (512, 1000, 6144),
])
def test_ragged_shapes(fs, dev, B, V, D):
    """Batch tails (B not a multiple of 128), vocabulary tails (V not a
    multiple of 16 / 256), partial k-blocks (D not a multiple of 64), several
    tiles per CTA (V / 152 > 256) and several batch tiles.  B = 16 / 17 and
    88 / 89 sit on the ring-depth boundaries of a single batch tile (6, 5 and
    4 stages), with several tiles per CTA so the last tile's parked noise is
    used too; B = 33, 64 / 65 and 96 / 97 on the accumulator-lane offsets
    (64, 32, 0) of a single batch tile.  Two batch tiles run the multicast
    pair below D = 4096 (B = 129, 130; B = 256 at D = 4032) and the pair MMA
    from it (B = 256 at D = 4096, 8192 and 65536: 64, 128 and 1024 k-blocks
    per tile); four batch tiles switch at D = 6144 (B = 512 at D = 6080 and
    6144)."""
    g = torch.Generator(device="cpu").manual_seed(B * 7919 + V * 31 + D)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * (1.5 / D ** 0.5)).to(torch.bfloat16).to(dev)
    run_and_check(fs, H, W, 0.9, 1000 + B, 3, "B=%d V=%d D=%d" % (B, V, D))


@pytest.mark.parametrize("B,D,form", [
    (64, 4096, 0), (100, 3584, 0), (384, 8192, 0),   # one or three batch tiles
    (256, 3584, 1), (512, 2304, 1), (512, 4096, 1),  # pairs below the D switch
    (256, 4096, 2), (256, 8192, 2), (512, 6144, 2), (1024, 8192, 2)])
def test_stage1_form_rule(fs, dev, B, D, form):
    """The launch form the library reports (and launches) for each shape:
    pairs only for an even number of batch tiles, the pair MMA from D = 4096
    with two batch tiles and from D = 6144 with more."""
    assert fs.fs_stage1_form(B, 128256, D) == form


def _random_shapes(n=48, seed=20261203):
    """Seeded (B, V, D) triples spread over the three launch forms: one batch
    tile, an odd number of batch tiles (unpaired), two and four batch tiles
    (paired: the multicast pair below the D switch, the pair MMA above it;
    half of the paired draws take D in 3584..8192).  D is a multiple of 8 (the call's own rule), V x D stays below 3e7 so
    that the oracle's rows take well under a second."""
    rng = np.random.default_rng(seed)
    spans = [(1, 128), (129, 256), (257, 384), (385, 512)]
    out = []
    for k in range(n):
        lo, hi = spans[k % len(spans)]
        B = int(rng.integers(lo, hi + 1))
        if k % 4 in (1, 3) and k % 8 >= 4:  # paired, near and above the form switch
            D = 8 * int(rng.integers(448, 1025))
        else:
            D = int(8 * max(1, round(float(np.exp(rng.uniform(0.0, np.log(1024)))))))
        vmax = max(1, min(60000, int(3e7 // D)))
        V = int(max(1, round(float(np.exp(rng.uniform(0.0, np.log(vmax)))))))
        out.append((B, V, D))
    return out


@pytest.mark.parametrize("k,B,V,D", [(k,) + s for k, s in enumerate(_random_shapes())])
def test_seeded_random_shapes(fs, dev, k, B, V, D):
    """Random shapes from a fixed seed: six rows (first, last, spread) of each
    against the oracle, alternately in the logits-store mode (logits compared
    too) and in the plain sampling mode, with a scalar or a per-row
    temperature."""
    g = torch.Generator(device="cpu").manual_seed(7000 + k)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * (2.0 / D ** 0.5)).to(torch.bfloat16).to(dev)
    T = (0.3 + 1.2 * torch.rand(B, generator=g)).to(dev) if k % 3 == 0 else 0.3 + 0.1 * (k % 12)
    run_and_check(fs, H, W, T, 500 + k, k, "random k=%d B=%d V=%d D=%d" % (k, B, V, D),
                  store=(k % 2 == 0), rows=spread_rows(B, 6))


@pytest.mark.parametrize("B,V,D,T,spread", [(64, 50000, 64, 0.05, 1.0), (200, 60000, 128, 1.0, 12.0),
                                             (256, 151936, 64, 0.8, 8.0), (3, 20011, 64, 0.01, 1.0)])
def test_peaked_logits(fs, dev, B, V, D, T, spread):
    """Logits so spread out (large scale, or a small temperature) that the
    per-element screen rejects almost every element: every row still matches
    the oracle, and the unfused path, which scans each row differently, agrees
    bit for bit.  A planted per-column bias (one column in 50 lifted) mimics
    the peaked distribution of real LM heads."""
    g = torch.Generator(device="cpu").manual_seed(B + V + int(100 * T))
    H = torch.randn((B, D), generator=g)
    H[:, D - 1] = 1.0
    W = torch.randn((V, D), generator=g) * (spread / D ** 0.5)
    lift = torch.rand(V, generator=g) < 0.02
    W[:, D - 1] = torch.where(lift, torch.full((V,), 4.0 * spread), torch.full((V,), -4.0 * spread))
    H = H.to(torch.bfloat16).to(dev)
    W = W.to(torch.bfloat16).to(dev)
    run_and_check(fs, H, W, T, 77 + B, 5, "peaked B=%d V=%d T=%g" % (B, V, T), store=False)
    fi, fsc, _ = fs.fs_sample_ex(H, W, temperature=T, seed=77 + B, offset=5)
    ui, usc, _ = fs.fs_sample_unfused(H, W, temperature=T, seed=77 + B, offset=5,
                                      y_dtype=fs.FS_DTYPE_F32)
    torch.cuda.synchronize()
    assert torch.equal(fi, ui) and torch.equal(fsc, usc)


@pytest.mark.parametrize("B,D", [(40, 128), (256, 128), (256, 6144)])
def test_per_row_temperatures_with_invalid_rows(fs, dev, B, D):
    """Invalid per-row temperatures give -1 / NaN for their rows only, in a
    single batch tile (B=40), in the multicast pair (B=256, D=128) and in the
    pair MMA (B=256, D=6144)."""
    V = 3000
    g = torch.Generator(device="cpu").manual_seed(4 + B + D)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    T = 0.5 + torch.rand(B, generator=g)
    T[3] = 0.0
    T[7] = -1.0
    T[11] = float("inf")
    T[19] = float("nan")
    T[23] = 1e-3
    T[29] = 1e3
    if B > 128:
        T[130] = 0.0     # in the peer CTA's batch tile
        T[255] = float("nan")
    run_and_check(fs, H, W, T.to(dev), 77, 1, "per-row T B=%d" % B)


def test_no_noise_ties_go_to_lowest_index(fs, dev):
    """Duplicated W rows give exact logit ties; with the noise off the lowest
    duplicate must win in every tile/partition arrangement."""
    B, V, D = 16, 20000, 64
    g = torch.Generator(device="cpu").manual_seed(9)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16)
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16)
    l = (H.float() @ W.float().T)
    top = l.argmax(dim=1)
    for b in range(B):  # copy each row's winner to several later positions
        for dst in (int(top[b]) + 1 + 997 * b % 5000, V - 1 - b):
            if dst < V and dst > int(top[b]):
                W[dst] = W[top[b]]
    idx, _ = run_and_check(fs, H.to(dev), W.to(dev), 1.0, 0, 0, "no-noise ties",
                           flags=fs.FS_FLAG_NO_NOISE)


def test_bigvocab_duplicates_small(fs, dev):
    B, V, D = 8, 26214, 64
    W = workloads.make_weights("bigvocab", V=V, D=D).to(dev)
    H = workloads.make_hidden("bigvocab", B, D=D).to(dev)
    run_and_check(fs, H, W, 1.0, 5, 0, "bigvocab-small noise")
    run_and_check(fs, H, W, 1.0, 5, 0, "bigvocab-small no-noise", flags=fs.FS_FLAG_NO_NOISE)


# ---------------------------------------------------------------- API consistency

def test_entry_points_agree_and_are_deterministic(fs, dev):
    B, V, D = 70, 30011, 192
    g = torch.Generator(device="cpu").manual_seed(21)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.08).to(torch.bfloat16).to(dev)
    T = (0.5 + torch.rand(B, generator=g)).to(dev)
    i1, s1 = fs.fs_sample(H, W, temperature=T, seed=3, offset=9)
    i2, s2, _ = fs.fs_sample_ex(H, W, temperature=T, seed=3, offset=9)
    ws = fs.workspace(B, V, D)
    fs.fs_stage1(H, W, ws, temperature=T, seed=3, offset=9)
    i3 = torch.empty(B, dtype=torch.int64, device=dev)
    s3 = torch.empty(B, dtype=torch.float32, device=dev)
    fs.fs_stage2(B, V, D, ws, temperature=T, out_idx=i3, out_score=s3)
    i4, s4, _ = fs.fs_sample_ex(H, W, temperature=T, seed=3, offset=9,
                                flags=fs.FS_FLAG_STORE_LOGITS)
    torch.cuda.synchronize()
    for i, s in ((i2, s2), (i3, s3), (i4, s4)):
        assert torch.equal(i1, i) and torch.equal(s1, s)
    # another offset changes the draw
    i5, _ = fs.fs_sample(H, W, temperature=T, seed=3, offset=10)
    assert not torch.equal(i1, i5)


def test_side_stream_and_workspace_growth(fs, dev):
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for B in (2, 300, 5):
            g = torch.Generator(device="cpu").manual_seed(B)
            H = torch.randn((B, 64), generator=g).to(torch.bfloat16).to(dev)
            W = (torch.randn((9000, 64), generator=g) * 0.1).to(torch.bfloat16).to(dev)
            outs.append((H, W, fs.fs_sample(H, W, temperature=1.0, seed=1, offset=2)))
    s.synchronize()
    for H, W, (idx, score) in outs:
        ref, _ = fs.fs_sample(H, W, temperature=1.0, seed=1, offset=2)
        assert torch.equal(idx, ref)


def test_host_buffer_entry(fs, dev):
    """fs_sample_host (H, T and the outputs in host memory) equals fs_sample on
    device copies bit for bit, with pinned and pageable buffers; back-to-back
    calls on one stream reuse the staging block in order."""
    B, V, D = 70, 30011, 192
    g = torch.Generator(device="cpu").manual_seed(33)
    Hs = [torch.randn((B, D), generator=g).to(torch.bfloat16) for _ in range(3)]
    W = (torch.randn((V, D), generator=g) * 0.08).to(torch.bfloat16).to(dev)
    T = 0.5 + torch.rand(B, generator=g)
    refs = [fs.fs_sample(H.to(dev), W, temperature=T.to(dev), seed=5, offset=k)
            for k, H in enumerate(Hs)]
    pinned = [H.pin_memory() for H in Hs]
    outs = [fs.fs_sample_host(H, W, temperature=T.pin_memory(), seed=5, offset=k)
            for k, H in enumerate(pinned)]
    torch.cuda.synchronize()
    for (ri, rs), (oi, os_) in zip(refs, outs):
        assert torch.equal(ri.cpu(), oi) and torch.equal(rs.cpu(), os_)
    # pageable host memory, scalar temperature, no score
    i_ref, _ = fs.fs_sample(Hs[0].to(dev), W, temperature=0.9, seed=6, offset=1)
    idx = torch.empty(B, dtype=torch.int64)
    fs.fs_sample_host(Hs[0], W, temperature=0.9, seed=6, offset=1, out_idx=idx, want_score=False)
    torch.cuda.synchronize()
    assert torch.equal(i_ref.cpu(), idx)
    # the tiny workload through host buffers against the oracle
    Wt = workloads.make_weights("tiny", device=dev)
    Ht = workloads.make_hidden("tiny", 4)
    seed, offset = workloads.sampling_seed("tiny", 4)
    ti, ts = fs.fs_sample_host(Ht.pin_memory(), Wt, temperature=1.0, seed=seed, offset=offset)
    torch.cuda.synchronize()
    assert fs.fs_get_device_status() == 0
    o_idx, o_best, o_second, _ = oracle.sample(bits(Ht), bits(Wt), np.ones(4, np.float32),
                                               seed, offset)
    compare_indices(ti.numpy(), o_idx, o_best, o_second, "host buffers")


def test_host_buffer_entry_mixed_upload_paths(fs, dev):
    """Page-locked inputs are uploaded by a kernel on the caller's stream,
    pageable ones by a copy on an internal stream; back-to-back calls that
    alternate between the two (no synchronisation in between) reuse the two
    device slots safely and each equals fs_sample on the same data."""
    g = torch.Generator(device="cpu").manual_seed(48)
    B, V, D = 40, 20011, 136
    W = (torch.randn((V, D), generator=g) * 0.09).to(torch.bfloat16).to(dev)
    Hs = [torch.randn((B, D), generator=g).to(torch.bfloat16) for _ in range(7)]
    T = 0.5 + torch.rand(B, generator=g)
    refs = [fs.fs_sample(H.to(dev), W, temperature=T.to(dev), seed=9, offset=k)[0].cpu()
            for k, H in enumerate(Hs)]
    outs = []
    for k, H in enumerate(Hs):
        pinned = k % 3 != 1
        Hk = H.pin_memory() if pinned else H.clone()
        Tk = T.pin_memory() if pinned else T.clone()
        idx = torch.empty(B, dtype=torch.int64).pin_memory()
        fs.fs_sample_host(Hk, W, temperature=Tk, seed=9, offset=k, out_idx=idx,
                          want_score=False)
        outs.append((Hk, Tk, idx))
    torch.cuda.synchronize()
    for k, (_, _, idx) in enumerate(outs):
        assert torch.equal(refs[k], idx), k


def test_host_buffer_entry_growth_and_graph_capture(fs, dev):
    """fs_sample_host grows its staging between batch sizes, and under CUDA
    graph capture (upload on the captured stream) replays to the same draw."""
    g = torch.Generator(device="cpu").manual_seed(44)
    W = (torch.randn((9001, 64), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    for B in (3, 200, 3, 129):
        H = torch.randn((B, 64), generator=g).to(torch.bfloat16)
        ref, rs = fs.fs_sample(H.to(dev), W, temperature=0.7, seed=8, offset=B)
        idx, sc = fs.fs_sample_host(H.pin_memory(), W, temperature=0.7, seed=8, offset=B)
        torch.cuda.synchronize()
        assert torch.equal(ref.cpu(), idx) and torch.equal(rs.cpu(), sc)
    B = 40
    H = torch.randn((B, 64), generator=g).to(torch.bfloat16).pin_memory()
    T = (0.5 + torch.rand(B, generator=g)).pin_memory()
    ref, rs = fs.fs_sample(H.to(dev), W, temperature=T.to(dev), seed=9, offset=4)
    s = torch.cuda.Stream()
    idx = torch.empty(B, dtype=torch.int64).pin_memory()
    sc = torch.empty(B, dtype=torch.float32).pin_memory()
    with torch.cuda.stream(s):  # warm-up: staging and workspace exist before capture
        fs.fs_sample_host(H, W, temperature=T, seed=9, offset=4, out_idx=idx, out_score=sc)
    s.synchronize()
    idx.fill_(-7)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fs.fs_sample_host(H, W, temperature=T, seed=9, offset=4, out_idx=idx, out_score=sc)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(ref.cpu(), idx) and torch.equal(rs.cpu(), sc)


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_graph_capture_of_fs_sample(fs, dev):
    """fs_sample captured into a CUDA graph after one call on the capture stream
    replays to the direct call's draw; on a fresh stream, capture refuses to
    grow the cached workspace (graph-owned memory must not enter the cache)."""
    g = torch.Generator(device="cpu").manual_seed(45)
    B, V, D = 24, 12011, 128
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    ref, rs = fs.fs_sample(H, W, temperature=0.9, seed=11, offset=3)
    s = torch.cuda.Stream()
    idx = torch.empty(B, dtype=torch.int64, device=dev)
    sc = torch.empty(B, dtype=torch.float32, device=dev)
    with torch.cuda.stream(s):
        fs.fs_sample(H, W, temperature=0.9, seed=11, offset=3, out_idx=idx, out_score=sc)
    s.synchronize()
    idx.fill_(-7)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fs.fs_sample(H, W, temperature=0.9, seed=11, offset=3, out_idx=idx, out_score=sc)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(ref, idx) and torch.equal(rs, sc)
    H_h = H.cpu().pin_memory()
    idx_h = torch.empty(B, dtype=torch.int64).pin_memory()
    fresh = torch.cuda.Stream()
    empty = torch.cuda.CUDAGraph()
    with torch.cuda.graph(empty, stream=fresh):
        with pytest.raises(fs.FSError, match="capture"):
            fs.fs_sample(H, W, temperature=0.9, seed=11, offset=3, out_idx=idx)
        with pytest.raises(fs.FSError, match="capture"):
            fs.fs_sample_host(H_h, W, temperature=0.9, seed=11, offset=3, out_idx=idx_h,
                              want_score=False)
    torch.cuda.synchronize()


def test_concurrent_host_threads(fs, dev):
    """Two host threads, each with its own stream, call fs_sample and
    fs_sample_host at the same time (ctypes releases the GIL): the library's
    caches are per (device, stream) and locked, so every result equals the
    sequential one."""
    import threading
    g = torch.Generator(device="cpu").manual_seed(46)
    B, V, D = 40, 20011, 128
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    Hs = [torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev) for _ in range(2)]
    refs = [[fs.fs_sample(Hs[t], W, temperature=0.8, seed=t, offset=k)[0] for k in range(20)]
            for t in range(2)]
    torch.cuda.synchronize()
    outs = [[None] * 20 for _ in range(2)]
    errors = []

    def worker(t):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream()
            H_h = Hs[t].cpu().pin_memory()
            with torch.cuda.stream(s):
                for k in range(20):
                    if k % 2:
                        outs[t][k] = fs.fs_sample_host(H_h, W, temperature=0.8, seed=t,
                                                       offset=k, want_score=False)[0]
                    else:
                        outs[t][k] = fs.fs_sample(Hs[t], W, temperature=0.8, seed=t,
                                                  offset=k)[0]
            s.synchronize()
        except Exception as e:  # reported in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(2):
        for k in range(20):
            assert torch.equal(refs[t][k].cpu(), outs[t][k].cpu()), (t, k)


def test_back_to_back_calls_overlap_safely(fs, dev):
    """Stage 1 is launched with programmatic dependent launch, so consecutive
    calls on one stream overlap their set-up.  A mixed sequence issued without
    any synchronisation must give exactly the results of the same calls run
    one by one with a synchronisation in between (workspace reuse, outputs
    consumed by the next call, a GEMM whose Y feeds the next call)."""
    g = torch.Generator(device="cpu").manual_seed(47)
    B, V, D = 48, 30011, 192
    W = (torch.randn((V, D), generator=g) * 0.08).to(torch.bfloat16).to(dev)
    Hs = [torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev) for _ in range(4)]
    bias = (torch.randn(V, generator=g) * 0.3).to(dev)
    ws = fs.workspace(B, V, D)

    def sequence(sync):
        out = []
        def step(x):
            out.append(x)
            if sync:
                torch.cuda.synchronize()
        for k in range(3):
            step(fs.fs_sample(Hs[k], W, temperature=0.8, seed=5, offset=k)[0].clone())
            step(fs.fs_sample_logprob(Hs[k + 1], W, temperature=1.1, seed=6, offset=k)[2].clone())
            fs.fs_stage1(Hs[k], W, ws, temperature=0.9, seed=7, offset=k)
            i2 = torch.empty(B, dtype=torch.int64, device=dev)
            fs.fs_stage2(B, V, D, ws, temperature=0.9, out_idx=i2)
            step(i2)
            step(fs.fs_sample_transformed(Hs[k + 1], W, bias=bias, softcap=20.0, temperature=0.7,
                                          seed=8, offset=k)[0].clone())
            Y = fs.fs_logits_gemm(Hs[k], W, y_dtype=fs.FS_DTYPE_F32)
            step(fs.fs_sample_from_logits(Y, temperature=0.8, seed=5, offset=k)[0].clone())
        torch.cuda.synchronize()
        return out

    ref = sequence(True)
    for _ in range(3):
        got = sequence(False)
        assert len(got) == len(ref)
        for i, (a, b) in enumerate(zip(ref, got)):
            assert torch.equal(a, b) or (a.is_floating_point() and
                                         torch.equal(torch.isnan(a), torch.isnan(b)) and
                                         torch.equal(a[~torch.isnan(a)], b[~torch.isnan(b)])), i
    # the unfused sample of a call equals the fused one (same noise, f32 logits)
    assert torch.equal(ref[0], ref[4])
    assert fs.fs_get_device_status() == 0


# ---------------------------------------------------------------- unfused comparator

@pytest.mark.parametrize("T", [0.8, 1e-3, 0.3, 50.0, "rows"])
@pytest.mark.parametrize("B,V,D,scale", [(65, 33000, 256, 0.08), (300, 20011, 64, 0.5),
                                         (7, 151936, 128, 0.02), (256, 30011, 192, 0.1),
                                         (256, 5003, 6144, 0.02)])
def test_unfused_f32_equals_fused(fs, dev, B, V, D, scale, T):
    """The unfused sampling pass evaluates every element's Gumbel; the fused
    epilogue screens elements that cannot win.  With f32 logits both must pick
    the same index with the same score, bit for bit, at any temperature."""
    g = torch.Generator(device="cpu").manual_seed(B + V)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * scale).to(torch.bfloat16).to(dev)
    if T == "rows":
        T = (torch.rand(B, generator=g) * 3.0 + 1e-3).to(dev)
    for off in (1, 2):
        fi, fsc, fl = fs.fs_sample_ex(H, W, temperature=T, seed=8, offset=off,
                                      flags=fs.FS_FLAG_STORE_LOGITS)
        ui, usc, Y = fs.fs_sample_unfused(H, W, temperature=T, seed=8, offset=off,
                                          y_dtype=fs.FS_DTYPE_F32)
        torch.cuda.synchronize()
        assert torch.equal(Y, fl)
        assert torch.equal(fi, ui)
        assert torch.equal(fsc, usc)


@pytest.mark.parametrize("B,V,D", [(9, 12345, 128), (256, 4099, 256), (256, 2053, 6144)])
def test_unfused_bf16_logits(fs, dev, B, V, D):
    """The logits GEMM (bf16 and f32 outputs) against the oracle's logits,
    in each launch form: one batch tile, the multicast pair, the pair MMA."""
    g = torch.Generator(device="cpu").manual_seed(6 + B + D)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.1).to(torch.bfloat16).to(dev)
    Y16 = fs.fs_logits_gemm(H, W, y_dtype=fs.FS_DTYPE_BF16)
    Y32 = fs.fs_logits_gemm(H, W, y_dtype=fs.FS_DTYPE_F32)
    torch.cuda.synchronize()
    o = oracle.logits(bits(H), bits(W)).astype(np.float64)
    assert np.abs(Y32.cpu().numpy() - o).max() <= LOGIT_TOL
    y16 = Y16.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y16 - o) <= LOGIT_TOL + np.abs(o) * 2.0 ** -8)
    assert torch.equal(Y16, Y32.to(torch.bfloat16))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,V", [(1, 7), (6, 8193), (33, 50000)])
def test_sample_from_materialised_logits(fs, dev, dtype, B, V):
    """The unfused sampling pass on seeded synthetic logits vs the oracle's
    full pass over the same logits."""
    g = torch.Generator(device="cpu").manual_seed(B * 13 + V)
    Y = (2.0 * torch.randn((B, V), generator=g)).to(dtype)
    T = (0.5 + torch.rand(B, generator=g))
    idx, score = fs.fs_sample_from_logits(Y.to(dev), temperature=T.to(dev), seed=42, offset=3)
    torch.cuda.synchronize()
    o_idx, o_best, o_second, _ = oracle.sample_from_logits(Y.float().numpy(), T.numpy(), 42, 3)
    compare_indices(idx.cpu().numpy(), o_idx, o_best, o_second, "logits %s B=%d V=%d" % (dtype, B, V))
    same = idx.cpu().numpy() == o_idx
    assert np.all(np.abs(score.cpu().numpy()[same] - o_best[same]) <= 4e-6 * np.abs(o_best[same]) + 2e-6)


# ---------------------------------------------------------------- full-size workloads

# (workload, B): one CTA per batch tile for B <= 128 and an odd number of
# batch tiles; for an even number, CTA pairs: multicast W for qwen B=256
# (D=3584) and bigvocab B=512 (D=2304), one M=256 MMA over both CTAs for
# llama3_70b (D=8192).
FULL = [("llama3_8b", 64), ("llama3_8b", 1), ("qwen", 256), ("qwen", 100),
        ("llama3_70b", 256), ("llama3_70b", 512), ("llama3_70b", 1024), ("bigvocab", 512),
        ("bigvocab", 64), ("bigvocab", 1)]
FULL_ROWS = 32


def spread_rows(B, n):
    """n rows of a batch of B: the first, the last and an even spread."""
    if B <= n:
        return np.arange(B)
    return np.unique(np.round(np.linspace(0, B - 1, n)).astype(np.int64))


@pytest.mark.parametrize("name,B", FULL)
def test_full_size_sampled_rows(fs, dev, name, B):
    """Each workload at full size through fs_sample_ex, the call the benchmark
    times: first in the logits-store mode (logits against the oracle's), then
    in the plain sampling mode that the timed calls run (the same launch
    configuration and kernel instantiation), both against the oracle on
    FULL_ROWS rows (first, last and spread); near-ties are counted."""
    W = workloads.make_weights(name, device=dev)
    H = workloads.make_hidden(name, B, device=dev)
    T = workloads.make_temperature(name, B, device=dev)
    seed, offset = workloads.sampling_seed(name, B)
    rows = spread_rows(B, FULL_ROWS)
    i_store, s_store = run_and_check(fs, H, W, T, seed, offset, "%s B=%d store" % (name, B),
                                     rows=rows)
    i_plain, s_plain = run_and_check(fs, H, W, T, seed, offset, "%s B=%d" % (name, B),
                                     store=False, rows=rows)
    # the two instantiations draw the same sample for every row of the batch
    assert torch.equal(i_store, i_plain) and torch.equal(s_store, s_plain)
    if name == "bigvocab":
        run_and_check(fs, H, W, T, seed, offset, "%s B=%d no-noise" % (name, B),
                      flags=fs.FS_FLAG_NO_NOISE, store=False, rows=rows)


def test_full_size_headline_every_row(fs, dev):
    """The benchmark's headline call (llama3_8b, B=64, offset 0 and the next
    decode offset): every row against the oracle."""
    name, B = "llama3_8b", 64
    W = workloads.make_weights(name, device=dev)
    H = workloads.make_hidden(name, B, device=dev)
    T = workloads.make_temperature(name, B, device=dev)
    seed, offset = workloads.sampling_seed(name, B)
    for off in (offset, offset + 1):
        run_and_check(fs, H, W, T, seed, off, "%s B=%d off=%d" % (name, B, off), store=False)


# ---------------------------------------------------------------- log-probability (log-mass)

@pytest.mark.parametrize("name,B,V,D", [("tiny", 4, None, None), ("qwen", 33, 20011, 128),
                                        ("llama3_8b", 64, 30000, 256), ("bigvocab", 200, 26214, 64),
                                        ("llama3_70b", 256, 9000, 128),
                                        ("llama3_70b", 256, 2053, 8192)])
def test_logprob_matches_oracle(fs, dev, name, B, V, D):
    """fs_sample_logprob: same samples as fs_sample_ex, and the sampled token's
    log-probability within 2 x the logits tolerance / T of the oracle's fp64
    log-softmax of the same token (a logit error moves both terms)."""
    W = workloads.make_weights(name, V=V, D=D).to(dev)
    H = workloads.make_hidden(name, B, D=D).to(dev)
    T = workloads.make_temperature(name, B, device=dev)
    seed, offset = workloads.sampling_seed(name, B)
    idx, score, lp = fs.fs_sample_logprob(H, W, temperature=T, seed=seed, offset=offset)
    i2, s2, _ = fs.fs_sample_ex(H, W, temperature=T, seed=seed, offset=offset)
    torch.cuda.synchronize()
    assert torch.equal(idx, i2) and torch.equal(score, s2)
    l32 = oracle.logits(bits(H), bits(W))
    Th = host_T(T, B)
    o_lp = oracle.logprob(l32, Th, idx.cpu().numpy())
    g_lp = lp.cpu().numpy().astype(np.float64)
    err = np.abs(g_lp - o_lp)
    tol = 2 * LOGIT_TOL / np.minimum(Th, 1.0) + 1e-4
    assert np.all(err <= tol), "max |d logprob| = %g" % err.max()
    assert np.all(g_lp <= 1e-6)
    print("[logprob %s B=%d] max |d| = %.2e" % (name, B, err.max()))


def test_logprob_invalid_rows_and_full_size(fs, dev):
    B, V, D = 9, 4099, 64
    g = torch.Generator(device="cpu").manual_seed(3)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.2).to(torch.bfloat16).to(dev)
    T = torch.full((B,), 0.8)
    T[2] = 0.0
    T[5] = float("nan")
    idx, score, lp = fs.fs_sample_logprob(H, W, temperature=T.to(dev), seed=1, offset=2)
    torch.cuda.synchronize()
    lp = lp.cpu().numpy()
    assert np.isnan(lp[2]) and np.isnan(lp[5]) and int(idx[2]) == -1
    assert np.all(np.isfinite(np.delete(lp, [2, 5])))
    # full-size decode row sample
    name, B = "llama3_8b", 64
    W = workloads.make_weights(name, device=dev)
    H = workloads.make_hidden(name, B, device=dev)
    idx, _, lp = fs.fs_sample_logprob(H, W, temperature=1.0, seed=7, offset=0)
    torch.cuda.synchronize()
    rows = np.array([0, 17, 63])
    l32 = oracle.logits(bits(H)[rows], bits(W))
    o = oracle.logprob(l32, 1.0, idx.cpu().numpy()[rows])
    err = np.abs(lp.cpu().numpy()[rows] - o)
    assert np.all(err <= 2 * LOGIT_TOL + 1e-4), err
    print("[logprob llama3_8b full] max |d| = %.2e" % err.max())


# ---------------------------------------------------------------- deterministic transforms

def _mask(rng, B, V, keep=0.7):
    words = (V + 31) // 32 + 1
    allowed = rng.random((B, words * 32)) < keep
    bits = np.zeros((B, words), dtype=np.uint64)
    for k in range(32):
        bits |= allowed[:, k::32].astype(np.uint64) << np.uint64(k)
    return bits.astype(np.uint32)


@pytest.mark.parametrize("B,V,D,softcap,use_bias,use_mask", [
    (37, 9001, 128, 0.0, True, False), (64, 40000, 64, 30.0, True, True),
    (5, 4099, 136, 10.0, False, True), (260, 20011, 64, 0.0, True, True),
    (256, 30011, 96, 25.0, True, True), (256, 3001, 6144, 20.0, True, True)])
def test_transforms_match_oracle(fs, dev, B, V, D, softcap, use_bias, use_mask):
    rng = np.random.default_rng(B + V)
    g = torch.Generator(device="cpu").manual_seed(B * 5 + V)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * (3.0 / D ** 0.5)).to(torch.bfloat16).to(dev)
    bias = (rng.standard_normal(V) * 2).astype(np.float32) if use_bias else None
    mask = _mask(rng, B, V) if use_mask else None
    T = torch.as_tensor(rng.uniform(0.5, 1.5, B).astype(np.float32))
    tb = torch.as_tensor(bias).to(dev) if use_bias else None
    tm = torch.as_tensor(mask.view(np.int32)).to(dev) if use_mask else None
    idx, score, lp = fs.fs_sample_transformed(H, W, bias=tb, softcap=softcap, allow_mask=tm,
                                              temperature=T.to(dev), seed=9, offset=4,
                                              want_logprob=True)
    # the instantiation without the log-mass draws the same sample
    i2, s2, _ = fs.fs_sample_transformed(H, W, bias=tb, softcap=softcap, allow_mask=tm,
                                         temperature=T.to(dev), seed=9, offset=4)
    torch.cuda.synchronize()
    assert torch.equal(idx, i2) and torch.equal(score, s2)
    l32 = oracle.logits(bits(H), bits(W))
    lx = oracle.transform_logits(l32, bias, softcap, mask)
    o_idx, o_best, o_second, _ = oracle.sample_from_logits(lx, T.numpy(), 9, 4)
    g_idx = idx.cpu().numpy()
    compare_indices(g_idx, o_idx, o_best, o_second, "transforms B=%d V=%d" % (B, V))
    same = g_idx == o_idx
    assert np.all(np.abs(score.cpu().numpy()[same] - o_best[same]) <= 1e-3)
    if use_mask:
        words = mask[np.arange(B), g_idx // 32]
        assert np.all((words >> (g_idx % 32).astype(np.uint32)) & 1), "a masked token was sampled"
    o_lp = oracle.logprob(lx, T.numpy(), g_idx)
    err = np.abs(lp.cpu().numpy() - o_lp)
    assert np.all(err <= 2 * LOGIT_TOL / 0.5 + 1e-4), err.max()
    print("[transforms B=%d V=%d] max |d logprob| = %.2e" % (B, V, err.max()))


def _random_paired_shapes(n=12, seed=77031):
    """Seeded paired shapes (two or four batch tiles, partial last tiles)
    with D from 3584 to 8192 (both pair forms, the pair MMA with its column
    hand-off) and a small V so that the oracle's full rows stay cheap."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        B = int(rng.integers(129, 257)) if k % 2 == 0 else int(rng.integers(385, 513))
        D = 8 * int(rng.integers(448, 1025))
        V = int(rng.integers(40, 700))
        out.append((B, V, D))
    return out


@pytest.mark.parametrize("k,B,V,D", [(k,) + s for k, s in enumerate(_random_paired_shapes())])
def test_seeded_random_paired_logprob_and_transforms(fs, dev, k, B, V, D):
    """Random paired shapes through the log-probability and transform modes
    (with and without the log-mass): samples and log-probabilities against
    the oracle on every row."""
    rng = np.random.default_rng(900 + k)
    g = torch.Generator(device="cpu").manual_seed(900 + k)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * (3.0 / D ** 0.5)).to(torch.bfloat16).to(dev)
    T = torch.as_tensor(rng.uniform(0.5, 1.5, B).astype(np.float32))
    l32 = oracle.logits(bits(H), bits(W))
    # log-probability mode
    idx, score, lp = fs.fs_sample_logprob(H, W, temperature=T.to(dev), seed=31 + k, offset=k)
    torch.cuda.synchronize()
    o_idx, o_best, o_second, _ = oracle.sample_from_logits(l32, T.numpy(), 31 + k, k)
    g_idx = idx.cpu().numpy()
    compare_indices(g_idx, o_idx, o_best, o_second, "logprob k=%d B=%d V=%d D=%d" % (k, B, V, D))
    err = np.abs(lp.cpu().numpy() - oracle.logprob(l32, T.numpy(), g_idx))
    assert np.all(err <= 2 * LOGIT_TOL / 0.5 + 1e-4), err.max()
    # transform modes
    bias = (rng.standard_normal(V) * 2).astype(np.float32)
    mask = _mask(rng, B, V)
    softcap = 20.0 if k % 3 else 0.0
    tb = torch.as_tensor(bias).to(dev)
    tm = torch.as_tensor(mask.view(np.int32)).to(dev)
    i1, s1, lp1 = fs.fs_sample_transformed(H, W, bias=tb, softcap=softcap, allow_mask=tm,
                                           temperature=T.to(dev), seed=57 + k, offset=2 * k,
                                           want_logprob=True)
    i2, s2, _ = fs.fs_sample_transformed(H, W, bias=tb, softcap=softcap, allow_mask=tm,
                                         temperature=T.to(dev), seed=57 + k, offset=2 * k)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(s1, s2)
    lx = oracle.transform_logits(l32, bias, softcap, mask)
    o_idx, o_best, o_second, _ = oracle.sample_from_logits(lx, T.numpy(), 57 + k, 2 * k)
    g_idx = i1.cpu().numpy()
    compare_indices(g_idx, o_idx, o_best, o_second, "transforms k=%d B=%d V=%d D=%d" % (k, B, V, D))
    live = g_idx >= 0
    err = np.abs(lp1.cpu().numpy()[live] - oracle.logprob(lx, T.numpy(), g_idx)[live])
    assert np.all(err <= 2 * LOGIT_TOL / 0.5 + 1e-4), err.max()


def test_zero_transforms_equal_plain_sampling_and_full_mask(fs, dev):
    B, V, D = 70, 30011, 192
    g = torch.Generator(device="cpu").manual_seed(77)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.08).to(torch.bfloat16).to(dev)
    i1, s1, _ = fs.fs_sample_transformed(H, W, temperature=0.9, seed=3, offset=5)
    i2, s2, _ = fs.fs_sample_ex(H, W, temperature=0.9, seed=3, offset=5)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(s1, s2)
    words = (V + 31) // 32
    m = torch.full((B, words), -1, dtype=torch.int32)
    m[4] = 0  # row 4: every token masked
    i3, s3, lp3 = fs.fs_sample_transformed(H, W, allow_mask=m.to(dev), temperature=0.9, seed=3,
                                           offset=5, want_logprob=True)
    torch.cuda.synchronize()
    assert int(i3[4]) == -1 and float(s3[4]) == float("-inf") and np.isnan(float(lp3[4]))
    keep = torch.ones(B, dtype=torch.bool)
    keep[4] = False
    assert torch.equal(i3[keep.to(dev)], i1[keep.to(dev)])


# ---------------------------------------------------------------- grouped sampling / shards

@pytest.mark.parametrize("B,V,D,cuts", [(6, 20000, 64, (4096, 12000)),
                                        (130, 30011, 96, (16, 20000)),
                                        (256, 3001, 6144, (1024,)),
                                        (64, 151936, 128, (75968,))])
def test_shards_and_grouped_combine(fs, dev, B, V, D, cuts):
    """Each shard's local sample (global indices, global noise) and log-mass
    match the oracle; merging the shards' candidates by score reproduces the
    unsharded sample (the pages' candidate exchange); the grouped combine
    matches the oracle's (group decisions in f32; near-ties counted)."""
    g = torch.Generator(device="cpu").manual_seed(B * 3 + V)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * (2.0 / D ** 0.5)).to(torch.bfloat16).to(dev)
    T = (0.6 + torch.rand(B, generator=g)).to(dev)
    seed, off = 4321, 9
    bounds = list(zip((0,) + cuts, cuts + (V,)))
    g_idx, g_sc, g_lm, o_idx, o_sc, o_lm = [], [], [], [], [], []
    Hb, Th = bits(H), host_T(T, B)
    for v0, v1 in bounds:
        i, sc, lm = fs.fs_sample_shard(H, W[v0:v1].contiguous(), v0, temperature=T, seed=seed,
                                       offset=off)
        torch.cuda.synchronize()
        oi, osc, olm, osec = oracle.sample_shard(Hb, bits(W[v0:v1].contiguous()), v0, Th, seed,
                                                 off)
        compare_indices(i.cpu().numpy(), oi, osc, osec, "shard [%d,%d)" % (v0, v1))
        assert np.all(np.abs(lm.cpu().numpy() - olm) <= 2 * LOGIT_TOL / 0.6 + 1e-4)
        g_idx.append(i); g_sc.append(sc); g_lm.append(lm)
        o_idx.append(oi); o_sc.append(osc); o_lm.append(olm)
    # candidate exchange: the best of the shards' candidates is the unsharded sample
    full_idx, full_sc, _ = fs.fs_sample_ex(H, W, temperature=T, seed=seed, offset=off)
    S = torch.stack(g_sc)
    k = torch.argmax(S, dim=0)
    merged = torch.stack(g_idx)[k, torch.arange(B, device=dev)]
    torch.cuda.synchronize()
    diff = (merged != full_idx).cpu().numpy()
    top2 = torch.topk(S, min(2, len(bounds)), dim=0).values.cpu().numpy()
    gap = top2[0] - top2[-1] if len(bounds) > 1 else np.full(B, np.inf)
    assert np.all(gap[diff] < NEAR_TIE), "shard merge differs from the unsharded sample"
    # grouped combine
    c_idx, c_grp = fs.fs_combine_groups(torch.stack(g_idx), torch.stack(g_lm), seed=777, offset=off)
    torch.cuda.synchronize()
    oc_idx, oc_grp, oc_best, oc_second = oracle.combine_groups(
        np.stack(o_idx), np.stack(o_lm), 777, off, want_scores=True)
    grp_near = (oc_best - oc_second) < NEAR_TIE
    gm = c_grp.cpu().numpy() != oc_grp
    assert not np.any(gm & ~grp_near), "group choice differs away from a near-tie"
    same = ~gm
    assert np.array_equal(c_idx.cpu().numpy()[same], np.stack([x.cpu().numpy() for x in g_idx])[c_grp.cpu().numpy()[same], np.arange(B)[same]])
    print("[grouped B=%d V=%d] group near-ties %d, mismatches %d" % (B, V, int(grp_near.sum()), int(gm.sum())))


def test_shard_at_the_top_of_the_index_range(fs, dev):
    """A ragged shard whose last row has global index 2^31 - 2, the largest
    the ABI accepts (offset + rows <= 2^31 - 1): local samples (global
    indices and noise) and log-masses against the oracle; one more row is
    refused."""
    B, Vs, D = 9, 5003, 64
    off0 = ((1 << 31) - Vs) // 16 * 16
    Vs = (1 << 31) - 1 - off0  # last global index 2^31 - 2
    g = torch.Generator(device="cpu").manual_seed(31)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((Vs, D), generator=g) * (2.0 / D ** 0.5)).to(torch.bfloat16).to(dev)
    i, sc, lm = fs.fs_sample_shard(H, W, off0, temperature=0.8, seed=5, offset=6)
    torch.cuda.synchronize()
    oi, osc, olm, osec = oracle.sample_shard(bits(H), bits(W), off0, host_T(0.8, B), 5, 6)
    compare_indices(i.cpu().numpy(), oi, osc, osec, "shard [%d, 2^31)" % off0)
    assert np.all(np.abs(lm.cpu().numpy() - olm) <= 2 * LOGIT_TOL / 0.8 + 1e-4)
    assert Vs % 16 != 0 and int(i.max()) <= (1 << 31) - 2 and int(i.min()) >= off0
    W2 = torch.zeros((Vs + 1, D), dtype=torch.bfloat16, device=dev)
    with pytest.raises(fs.FSError):
        fs.fs_sample_shard(H, W2, off0, temperature=0.8, seed=5, offset=6)


# ---------------------------------------------------------------- exactness of the law, edge sizes

def _chisq_p(counts, probs):
    import scipy.stats
    exp = probs * counts.sum()
    small = exp < 5
    if small.any():
        counts = np.append(counts[~small], counts[small].sum())
        exp = np.append(exp[~small], exp[small].sum())
    return scipy.stats.chisquare(counts, exp).pvalue


@pytest.mark.parametrize("V,T", [(64, 0.5), (64, 1.0), (64, 1.5), (2, 1.0), (8, 0.7)])
def test_gpu_samples_follow_softmax(fs, dev, V, T):
    """10^5 rows with the same hidden state (so the same logits) draw
    independent noise; the fused kernel's token frequencies must match
    softmax(l/T) of those logits (chi-squared, p > 0.01)."""
    import scipy.special
    N, D = 100_000, 64
    g = torch.Generator(device="cpu").manual_seed(V * 10 + int(10 * T))
    h = torch.randn((1, D), generator=g)
    H = h.expand(N, D).contiguous().to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.25).to(torch.bfloat16).to(dev)
    idx, _ = fs.fs_sample(H, W, temperature=T, seed=0xA11CE + V, offset=0)
    torch.cuda.synchronize()
    counts = np.bincount(idx.cpu().numpy(), minlength=V).astype(np.float64)
    l32 = oracle.logits(bits(H[:1]), bits(W))[0]
    lt = (l32 * (np.float32(1) / np.float32(T))).astype(np.float64)
    p = _chisq_p(counts, scipy.special.softmax(lt))
    print("[law V=%d T=%g] p = %.3f" % (V, T, p))
    assert p > 0.01


def test_edge_sizes(fs, dev):
    """V = 1; a 2^20-row batch; a 2^21-entry vocabulary (indices beyond 2^20)."""
    g = torch.Generator(device="cpu").manual_seed(99)
    # V = 1: every valid row samples token 0
    H = torch.randn((300, 16), generator=g).to(torch.bfloat16).to(dev)
    W = torch.randn((1, 16), generator=g).to(torch.bfloat16).to(dev)
    idx, _ = fs.fs_sample(H, W, temperature=1.0, seed=1, offset=0)
    torch.cuda.synchronize()
    assert torch.all(idx == 0)
    # large batch
    B, V, D = 1 << 20, 40, 64
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.2).to(torch.bfloat16).to(dev)
    rows = np.array([0, 1, 777, B // 2, B - 2, B - 1])
    run_and_check(fs, H, W, 0.8, 5, 6, "B=2^20", store=False, rows=rows)
    # large vocabulary
    B, V, D = 3, 1 << 21, 16
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.5).to(torch.bfloat16).to(dev)
    run_and_check(fs, H, W, 1.0, 7, 8, "V=2^21", store=False)


def test_maximum_batch_and_hidden_size(fs, dev):
    """B = 2^24 and D = 2^20, the largest the ABI accepts (each with a small
    other dimension): sampled rows against the oracle, among them the last
    row of the batch; one more row or 8 more columns are refused."""
    g = torch.Generator(device="cpu").manual_seed(2024)
    # B = 2^24: 131072 batch tiles in CTA pairs, one 24-row vocabulary tile
    B, V, D = 1 << 24, 24, 8
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.6).to(torch.bfloat16).to(dev)
    rows = np.array([0, 1, 129, 1 << 23, B - 2, B - 1])
    run_and_check(fs, H, W, 1.1, 21, 22, "B=2^24", store=False, rows=rows)
    with pytest.raises(fs.FSError):
        fs.fs_sample(torch.zeros((B + 1, D), dtype=torch.bfloat16, device=dev), W)
    del H
    # D = 2^20: 16384 k-blocks per tile, W rows of 2 MB
    B, V, D = 3, 40, 1 << 20
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * (1.0 / D ** 0.5)).to(torch.bfloat16).to(dev)
    run_and_check(fs, H, W, 0.5, 23, 24, "D=2^20")
    with pytest.raises(fs.FSError):
        fs.fs_sample(torch.zeros((B, D + 8), dtype=torch.bfloat16, device=dev),
                     torch.zeros((V, D + 8), dtype=torch.bfloat16, device=dev))
    torch.cuda.empty_cache()


def test_maximum_vocabulary(fs, dev):
    """V = 2^31 - 1, the largest vocabulary the ABI accepts: 34 GB of W at
    D = 8, a 14 M-row partition per CTA (55 K tiles).  Every row of W is zero
    except two whose logit is 64, one of them the very last row (inside the
    ragged last 16-row unit).  Their scores (>= 61) beat every other element
    (l + g <= 16.7), so the sample is whichever of the two draws the larger
    Gumbel.  The oracle draws those two Gumbels one by one and decides; over
    eight offsets each token wins at least once, and every decision and
    winning score match."""
    V, D = (1 << 31) - 1, 8
    hot = (1000, V - 1)
    seed = 0x5EED7777
    W = torch.zeros((V, D), dtype=torch.bfloat16, device=dev)
    try:
        for v in hot:
            W[v, 0] = 8.0
        H = torch.zeros((1, D), dtype=torch.bfloat16, device=dev)
        H[0, 0] = 8.0
        wins = set()
        for off in range(8):
            idx, score = fs.fs_sample(H, W, temperature=1.0, seed=seed, offset=off)
            torch.cuda.synchronize()
            assert fs.fs_get_device_status() == 0
            s = [np.float32(np.float32(64.0) + np.float32(oracle.gumbel(seed, off, 0, v)))
                 for v in hot]
            expect = hot[0] if s[0] >= s[1] else hot[1]
            got = int(idx[0])
            if abs(float(s[0]) - float(s[1])) >= NEAR_TIE:
                assert got == expect, "offset %d: sampled %d, oracle %d" % (off, got, expect)
            else:
                assert got in hot
            assert abs(float(score[0]) - float(max(s))) <= 2e-5
            wins.add(got)
        assert wins == set(hot)
    finally:
        del W
        torch.cuda.empty_cache()


def test_huge_batch_with_large_vocabulary(fs, dev):
    """B = 19201 (151 batch tiles, the last holding one row) and V = 3,200,011:
    one vocabulary partition per batch tile, so each CTA streams all of W in
    12,500 balanced tiles.  Sampled rows against the oracle, among them the
    single row of the last batch tile."""
    B, V, D = 19201, 3_200_011, 8
    g = torch.Generator(device="cpu").manual_seed(4242)
    H = torch.randn((B, D), generator=g).to(torch.bfloat16).to(dev)
    W = (torch.randn((V, D), generator=g) * 0.7).to(torch.bfloat16).to(dev)
    rows = np.array([0, 1, 127, 128, 9600, 19199, 19200])
    run_and_check(fs, H, W, 0.9, 11, 12, "B=%d V=%d" % (B, V), store=False, rows=rows)
