"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Every comparison is element by element on the same seeded inputs, within
|dy| <= 2^-7 |y_ref| + 1e-3; the exactness pins (one-hot weights, small
integer operands, zero K padding, TMA vs realigning loader) are bitwise.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import compare, to_dev, y_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines
    pytest.skip("needs a CUDA device", allow_module_level=True)

import fp8_channel_scaled_gb300 as fg  # noqa: E402
from fp8_channel_scaled_gb300 import Options, PATH_DECODE, PATH_MAIN  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_channel_scaled_gb300 import build
    build.build()
    fg.lib()
    yield
    assert fg.fp8_gemm_check_device_error() == 0


def run(x, w, s, options=None, y=None):
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    if y is None:
        y = torch.empty((x.shape[0], w.shape[0]), dtype=torch.bfloat16, device="cuda")
    if options is None:
        fg.fp8_gemm_scaled(xd, wd, sd, y)
    else:
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, options)
    fg.check_device_error()
    return y_bits(y)


def check_full(x, w, s, options=None, what=""):
    got = run(x, w, s, options)
    ref = oracle.linear(x, w, s)
    return compare(got, ref, what)


# ------------------------------------------------------------------ small workload
def test_small_workload_full():
    x, w, s = synth.workload_inputs("small")
    p = fg.plan(*x.shape[:1], w.shape[0], x.shape[1])
    assert p.path == PATH_DECODE and p.launches == 1
    check_full(x, w, s, what="small")


@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
def test_small_workload_both_paths(path):
    x, w, s = synth.workload_inputs("small")
    check_full(x, w, s, Options(path=path), what=f"small path {path}")


# ------------------------------------------------------------------ main path shapes and tails
MAIN_SHAPES = [
    (128, 256, 128), (256, 512, 1024), (129, 136, 256), (200, 300, 520), (65, 8, 16),
    (384, 264, 4127 // 8), (300, 257, 17), (130, 129, 129), (1, 1, 1), (77, 1000, 33),
    (640, 1280, 4096),
]


@pytest.mark.parametrize("M,N,K", MAIN_SHAPES)
@pytest.mark.parametrize("ctas", [1, 2])
def test_main_path_shapes(M, N, K, ctas):
    x, w, s = synth.make_inputs(M, N, K, seed=M * 7 + N * 3 + K)
    check_full(x, w, s, Options(path=PATH_MAIN, mma_ctas=ctas), what=f"main {M}x{N}x{K} ctas={ctas}")


@pytest.mark.parametrize("bn", [64, 128, 160, 192, 224, 256])
def test_main_path_tiles(bn):
    x, w, s = synth.make_inputs(300, 520, 640, seed=5)
    check_full(x, w, s, Options(path=PATH_MAIN, tile_n=bn, mma_ctas=1), what=f"main bn={bn}")


def test_narrow_tiles_for_mid_m():
    # 129-256 rows with few N blocks: 64-wide one-CTA tiles (twice the CTAs of
    # 128-wide ones); the CTA-pair kernel has no 64-wide tile
    p = fg.plan(256, 4096, 4096)
    assert (p.path, p.tile_m, p.tile_n, p.cluster) == (PATH_MAIN, 128, 64, 1)
    with pytest.raises(fg.FP8GemmError):
        fg.plan(256, 4096, 4096, Options(path=PATH_MAIN, mma_ctas=2, tile_n=64))
    x, w, s = synth.make_inputs(200, 4100, 700, seed=8)
    check_full(x, w, s, what="mid-M auto plan")


PAIR_SHAPES = [
    (256, 256, 256), (512, 448, 1024), (257, 300, 520), (129, 136, 128), (1000, 1000, 4096),
    (300, 257, 17 * 16), (64, 512, 256),
]


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
def test_cta_pair_tiles(M, N, K):
    x, w, s = synth.make_inputs(M, N, K, seed=M + 3 * N + 7 * K)
    p = fg.plan(M, N, K, Options(path=PATH_MAIN, mma_ctas=2))
    assert p.tile_m == 256 and p.cluster == 2 and p.grid % 2 == 0
    check_full(x, w, s, Options(path=PATH_MAIN, mma_ctas=2), what=f"pair {M}x{N}x{K}")


@pytest.mark.parametrize("bn", [128, 160, 192, 224, 256])
def test_cta_pair_tile_widths(bn):
    x, w, s = synth.make_inputs(600, 1000, 640, seed=bn)
    check_full(x, w, s, Options(path=PATH_MAIN, mma_ctas=2, tile_n=bn), what=f"pair bn={bn}")


def test_cta_pair_equals_single_cta_on_exact_sums():
    # integer operands: every fp32 partial sum is exact, so both tile kinds
    # must give identical bits (and equal the oracle's)
    codes = synth.quantize_e4m3(np.arange(-16, 17, dtype=np.float64))
    rng = np.random.default_rng(9)
    M, N, K = 384, 448, 2048
    x = rng.choice(codes, (M, K)).astype(np.uint8)
    w = rng.choice(codes, (N, K)).astype(np.uint8)
    s = (2.0 ** -rng.integers(0, 12, N)).astype(np.float32)
    a = run(x, w, s, Options(path=PATH_MAIN, mma_ctas=2))
    b = run(x, w, s, Options(path=PATH_MAIN, mma_ctas=1))
    assert np.array_equal(a, b)
    assert np.array_equal(a, oracle.linear(x, w, s))


@pytest.mark.parametrize("M,N,K,bn", [
    (512, 1024, 128, 256), (300, 520, 256, 224), (1000, 2000, 1000, 0), (256, 777, 384, 192),
    (768, 640, 3072, 128), (2048, 4096, 3001, 0), (600, 900, 700, 160),
])
def test_eight_epilogue_warps_match_four_bitwise(M, N, K, bn):
    # Pair tiles whose epilogue is split over eight warps (two per TMEM lane
    # quarter, each half the columns) store exactly what four warps store
    x, w, s = synth.make_inputs(M, N, K, seed=M + K)
    o8 = Options(path=PATH_MAIN, mma_ctas=2, tile_n=bn, epilogue_warps=8)
    o4 = Options(path=PATH_MAIN, mma_ctas=2, tile_n=bn, epilogue_warps=4)
    p8 = fg.plan(M, N, K, options=o8)
    assert p8.epilogue_warps == 8 and p8.threads == 384
    y8 = run(x, w, s, o8)
    compare(y8, oracle.linear(x, w, s), f"eight epilogue warps {M}x{N}x{K}")
    assert np.array_equal(y8, run(x, w, s, o4))


def test_short_k_plans_take_eight_epilogue_warps():
    assert fg.plan(8192, 8192, 128).epilogue_warps == 8
    assert fg.plan(8192, 8192, 1024).epilogue_warps == 8
    assert fg.plan(4096, 4096, 4096).epilogue_warps == 4
    assert fg.plan(512, 4096, 1024).epilogue_warps == 4  # one tile per pair
    assert fg.plan(4096, 4096, 1024, options=Options(split_tail=True)).epilogue_warps == 4
    with pytest.raises(fg.FP8GemmError):
        fg.plan(4096, 4096, 1024, options=Options(mma_ctas=2, epilogue_warps=6))


@pytest.mark.parametrize("bn", [128, 224, 256])
def test_main_path_realigning_loader(bn):
    x, w, s = synth.make_inputs(300, 520, 640, seed=5)
    check_full(x, w, s, Options(path=PATH_MAIN, tile_n=bn, force_realign=True),
               what=f"main realign bn={bn}")


@pytest.mark.parametrize("M,N,K", [(130, 264, 4127), (256, 300, 17), (129, 1000, 1000)])
def test_repitch_equals_in_kernel_loader_bitwise(M, N, K):
    x, w, s = synth.make_inputs(M, N, K, seed=K)
    p = fg.plan(M, N, K, Options(path=PATH_MAIN))
    assert p.repitch == 1 and p.launches == 2
    assert p.workspace_bytes >= M * ((K + 15) // 16 * 16) + N * ((K + 15) // 16 * 16)
    # no split tail: the in-kernel loader runs on one-CTA tiles, whose fp32
    # sums follow K in the same order as unsplit pair tiles
    a = run(x, w, s, Options(path=PATH_MAIN))
    b = run(x, w, s, Options(path=PATH_MAIN, no_workspace=True))
    assert np.array_equal(a, b)
    compare(a, oracle.linear(x, w, s), f"repitch {M}x{N}x{K}")
    compare(run(x, w, s, Options(path=PATH_MAIN, split_tail=True)), oracle.linear(x, w, s),
            f"repitch split {M}x{N}x{K}")


def test_caller_workspace():
    M, N, K = 200, 264, 4127
    x, w, s = synth.make_inputs(M, N, K, seed=2)
    need = fg.fp8_gemm_workspace_bytes(torch.cuda.current_device(), M, N, K)
    assert need > 0
    ws = torch.full((need + 512,), 0xAB, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    got = run(x, w, s, Options(workspace=base, workspace_bytes=need))
    compare(got, oracle.linear(x, w, s), "caller workspace")
    # a workspace that is too small is refused before anything runs
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, Options(workspace=base, workspace_bytes=need - 256))
    assert e.value.status == 1
    # aligned operands need no repitch workspace (only the split tail's, if any)
    assert fg.fp8_gemm_workspace_bytes(torch.cuda.current_device(), M, N, 4096) == 0


# ------------------------------------------------------------------ split tail (pair tiles)
def pairs_on_device():
    return fg.plan(4096, 4096, 4096, Options(path=PATH_MAIN, mma_ctas=2, tile_n=256)).grid // 2


def split_shapes():
    """Shapes whose last wave is split: no full wave, one full wave plus a
    few tiles, a ragged M/N/K edge, and few K blocks per tile."""
    P = pairs_on_device()
    return [
        (768, 2048, 1024),            # 24 tiles < P: the whole problem is tail
        (256 * ((P + 4) // 8 + 1), 2048, 512),  # one full wave, then a short tail
        (1000, 1500, 1000),           # ragged M, N and K (repitch + split)
        (512, 512, 256),              # 2 K blocks per tile: tiny segments
        (2048, 4096, 4096),
    ]


@pytest.mark.parametrize("case", range(5))
def test_split_tail_matches_oracle(case):
    M, N, K = split_shapes()[case]
    opts = Options(path=PATH_MAIN, mma_ctas=2, tile_n=256, split_tail=True)
    p = fg.plan(M, N, K, opts)
    assert p.split_tiles > 0 and p.tail_workers > p.split_tiles, p
    assert p.tail_workers <= 2 * p.split_tiles
    x, w, s = synth.make_inputs(M, N, K, seed=M + N + K)
    check_full(x, w, s, opts, what=f"split {M}x{N}x{K}")


def test_split_tail_exact_sums_and_determinism():
    # integer operands: the split sums are exact, so split and unsplit tiles
    # agree bitwise; and a split call gives the same bits every time
    codes = synth.quantize_e4m3(np.arange(-16, 17, dtype=np.float64))
    rng = np.random.default_rng(11)
    M, N, K = 768, 2048, 1024
    x = rng.choice(codes, (M, K)).astype(np.uint8)
    w = rng.choice(codes, (N, K)).astype(np.uint8)
    s = (2.0 ** -rng.integers(0, 12, N)).astype(np.float32)
    opts = Options(path=PATH_MAIN, mma_ctas=2, tile_n=256, split_tail=True)
    assert fg.plan(M, N, K, opts).split_tiles > 0
    a = run(x, w, s, opts)
    b = run(x, w, s, Options(path=PATH_MAIN, mma_ctas=2, tile_n=256))
    assert fg.plan(M, N, K, Options(path=PATH_MAIN, mma_ctas=2, tile_n=256)).split_tiles == 0
    assert np.array_equal(a, b)
    assert np.array_equal(a, oracle.linear(x, w, s))
    x2, w2, s2 = synth.make_inputs(M, N, K, seed=12)
    r1 = run(x2, w2, s2, opts)
    r2 = run(x2, w2, s2, opts)
    assert np.array_equal(r1, r2)


def test_split_tail_caller_workspace_and_stale_flags():
    # the caller's workspace holds leftovers of an earlier call; the flags are
    # matched against a per-call value, so the second call must not take the
    # first call's partial sums
    M, N, K = 768, 2048, 1024
    opts = Options(path=PATH_MAIN, mma_ctas=2, tile_n=256, split_tail=True)
    need = fg.fp8_gemm_workspace_bytes(torch.cuda.current_device(), M, N, K, opts)
    assert need > 0
    ws = torch.full((need + 512,), 0xFF, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    o2 = Options(path=PATH_MAIN, mma_ctas=2, tile_n=256, split_tail=True, workspace=base,
                 workspace_bytes=need)
    x, w, s = synth.make_inputs(M, N, K, seed=21)
    compare(run(x, w, s, o2), oracle.linear(x, w, s), "split caller ws 1")
    x2, w2, s2 = synth.make_inputs(M, N, K, seed=22)
    compare(run(x2, w2, s2, o2), oracle.linear(x2, w2, s2), "split caller ws 2")
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    small = Options(path=PATH_MAIN, mma_ctas=2, tile_n=256, split_tail=True, workspace=base,
                    workspace_bytes=need - 256)
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, small)
    assert e.value.status == 1
    # without any workspace the last wave runs unsplit
    assert fg.plan(M, N, K, Options(path=PATH_MAIN, mma_ctas=2, tile_n=256, split_tail=True,
                                    no_workspace=True)).split_tiles == 0
    # and it is off unless asked for
    assert fg.plan(M, N, K, Options(path=PATH_MAIN, mma_ctas=2, tile_n=256)).split_tiles == 0


def test_split_tail_back_to_back_on_one_stream():
    # consecutive split calls share nothing but the stream; each must see its
    # own partial sums (and the next call may start while this one drains)
    M, N, K = 768, 2048, 1024
    opts = Options(path=PATH_MAIN, mma_ctas=2, tile_n=256, split_tail=True)
    ins = [synth.make_inputs(M, N, K, seed=40 + i) for i in range(4)]
    dev = [(to_dev(x), to_dev(w), to_dev(s)) for x, w, s in ins]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in ins]
    for (xd, wd, sd), y in zip(dev, ys):
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, opts)
    fg.check_device_error()
    for (x, w, s), y in zip(ins, ys):
        compare(y_bits(y), oracle.linear(x, w, s), "back to back")


# ------------------------------------------------------------------ decode path shapes and tails
DECODE_SHAPES = [
    (1, 128, 128), (5, 136, 256), (32, 1024, 2048), (33, 1000, 1000), (64, 384, 4096),
    (17, 257, 4127), (32, 128, 8192), (100, 256, 512), (2, 8, 16),
    (129, 384, 1024), (200, 1000, 2048), (256, 640, 4096), (256, 136, 4127),
]


@pytest.mark.parametrize("M,N,K", DECODE_SHAPES)
def test_decode_path_shapes(M, N, K):
    x, w, s = synth.make_inputs(M, N, K, seed=M + N + K)
    check_full(x, w, s, Options(path=PATH_DECODE), what=f"decode {M}x{N}x{K}")


@pytest.mark.parametrize("M", [150, 192])
def test_mid_m_decode_path_and_its_no_workspace_fallback(M):
    # 129-192 rows (N <= 8192) take the decode kernel with x padded to 256
    # rows; that kernel has no realigning loader, so with no_workspace and
    # unaligned rows the plan moves to the tile kernel's loader
    N, K = 640, 4127
    x, w, s = synth.make_inputs(M, N, K, seed=M)
    p = fg.plan(M, N, K)
    assert p.path == PATH_DECODE and p.tile_n == 256 and p.repitch == 1
    check_full(x, w, s, what=f"mid-M {M} decode")
    p2 = fg.plan(M, N, K, options=Options(no_workspace=True))
    assert p2.path == PATH_MAIN and p2.realign == 1
    check_full(x, w, s, Options(no_workspace=True), what=f"mid-M {M} no workspace")


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
def test_decode_splits(splits):
    x, w, s = synth.make_inputs(32, 640, 2048, seed=splits)
    check_full(x, w, s, Options(path=PATH_DECODE, splits=splits), what=f"splits {splits}")


@pytest.mark.parametrize("M,N,K,kbs,stages,splits", [
    (32, 4096, 4096, 2, 5, 1), (32, 4096, 4096, 2, 5, 2), (32, 4096, 4096, 4, 2, 4),
    (17, 1000, 2048, 2, 4, 2), (1, 256, 1024, 4, 2, 1), (32, 640, 512, 2, 5, 2),
    (64, 1024, 2048, 4, 2, 2), (50, 300, 1024, 2, 4, 1), (32, 128, 256, 2, 5, 1),
    (100, 512, 1024, 2, 3, 2), (128, 384, 2048, 2, 3, 4), (200, 256, 512, 2, 2, 1),
])
def test_decode_several_k_blocks_per_stage(M, N, K, kbs, stages, splits):
    # Stages of 2 or 4 K blocks read with 3-D boxes (one per operand and
    # stage) land as ordinary K-major tiles: every output equals the oracle's
    # within the tolerance, with one split (outputs stored straight from
    # tensor memory) or several (cluster reduction)
    x, w, s = synth.make_inputs(M, N, K, seed=M * 7 + kbs)
    o = Options(path=PATH_DECODE, tile_n=kbs, stages=stages, splits=splits)
    p = fg.plan(M, N, K, o)
    assert p.kblocks_per_stage == kbs and p.stages == stages and p.splits == splits
    check_full(x, w, s, o, what=f"decode {M}x{N}x{K} kbs {kbs} stages {stages} splits {splits}")


@pytest.mark.parametrize("kbs,stages", [(2, 5), (4, 2)])
def test_decode_k_block_grouping_keeps_the_accumulation_order(kbs, stages):
    # one split accumulates the K blocks in order in one accumulator, however
    # many of them a stage holds: bitwise the same as one K block per stage
    M, N, K = 32, 2048, 4096
    x, w, s = synth.make_inputs(M, N, K, seed=61)
    a = run(x, w, s, Options(path=PATH_DECODE, tile_n=kbs, stages=stages, splits=1))
    b = run(x, w, s, Options(path=PATH_DECODE, tile_n=1, stages=4, splits=1))
    assert np.array_equal(a, b)
    compare(a, oracle.linear(x, w, s), f"kbs {kbs} single split")


def test_decode_workload_plan_and_k_block_rules():
    p = fg.plan(32, 8192, 8192)
    assert p.path == PATH_DECODE and p.kblocks_per_stage == 2 and p.stages == 5 and p.splits == 2
    assert fg.plan(32, 14336, 4096).splits == 1
    p = fg.plan(64, 4096, 4096)
    assert p.kblocks_per_stage == 2 and p.stages == 4 and p.splits == 4
    p = fg.plan(128, 8192, 8192)
    assert p.path == PATH_DECODE and p.kblocks_per_stage == 2 and p.stages == 3 and p.splits == 2
    # several K blocks per stage need K % 128 == 0: otherwise nothing is built
    with pytest.raises(fg.FP8GemmError) as e:
        fg.plan(32, 1024, 4100, Options(path=PATH_DECODE, tile_n=2))
    assert e.value.status == 6
    with pytest.raises(fg.FP8GemmError) as e:
        fg.plan(32, 1024, 4096, Options(path=PATH_DECODE, tile_n=3))
    assert e.value.status == 1
    # small weights keep one K block per stage
    assert fg.plan(32, 128, 256).kblocks_per_stage == 1


@pytest.mark.parametrize("M", [8, 40, 128])
def test_decode_realign(M):
    x, w, s = synth.make_inputs(M, 384, 1040, seed=M)
    check_full(x, w, s, Options(path=PATH_DECODE, force_realign=True), what=f"decode realign M={M}")


# ------------------------------------------------------------------ seeded random sweep
def _random_cases(n=28, seed=20261202):
    """Shapes and plan options drawn once from a fixed seed: sizes with
    every residue against the tile widths, the 16-byte K pitch and the
    128-byte K block, on every path and tile kind the planner can pick."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for i in range(n):
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 1300))
        K = int(rng.integers(1, 2200))
        kind = i % 7
        if kind == 0:
            opts = None
        elif kind == 1:
            opts = dict(path=PATH_MAIN, mma_ctas=1, tile_n=int(rng.choice([128, 160, 192, 224, 256])))
        elif kind == 2:
            opts = dict(path=PATH_MAIN, mma_ctas=2, tile_n=int(rng.choice([128, 160, 192, 224, 256])))
        elif kind == 3:
            opts = dict(path=PATH_MAIN, mma_ctas=2, split_tail=True)
        elif kind == 4:
            M = int(rng.integers(1, 129))
            opts = dict(path=PATH_DECODE, splits=int(rng.integers(1, 9)))
        elif kind == 5:
            opts = dict(path=PATH_MAIN, no_workspace=True)
        else:
            M = int(rng.integers(1, 129))
            opts = dict(path=PATH_DECODE)
        cases.append((M, N, K, opts, int(rng.integers(0, 2 ** 31))))
    return cases


@pytest.mark.parametrize("M,N,K,opts,seed", _random_cases())
def test_random_shapes_and_options(M, N, K, opts, seed):
    x, w, s = synth.make_inputs(M, N, K, seed=seed)
    o = None if opts is None else Options(**opts)
    if o is not None and o.path == PATH_DECODE and o.splits > max(1, (K + 127) // 128):
        o.splits = 0  # more splits than K blocks: let the planner choose
    check_full(x, w, s, o, what=f"random {M}x{N}x{K} {opts}")


# ------------------------------------------------------------------ maximum sizes
@pytest.mark.parametrize("N,ctas", [(16384, 2), (16384, 1), (16383, 2)])
def test_output_larger_than_2gib(N, ctas):
    # y holds more than 2^31 bytes, so every store path (TMA store, 16-byte
    # stores of one-CTA tiles, element stores when N % 8 != 0) must index it
    # with 64-bit offsets; rows around byte offset 2^31 and the last rows are
    # checked against the oracle.
    M, K = 70000, 32
    assert M * N * 2 > 2 ** 31
    x, w, s = synth.make_inputs(M, N, K, seed=77)
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fg.fp8_gemm_scaled_ex(xd, wd, sd, y, Options(path=PATH_MAIN, mma_ctas=ctas))
    fg.check_device_error()
    edge = (2 ** 31) // (2 * N)
    rng = np.random.default_rng(78)
    rows = np.unique(np.concatenate([[0, edge - 1, edge, edge + 1, M - 2, M - 1],
                                     rng.integers(0, M, 10)]))
    got = y_bits(y[torch.from_numpy(rows).cuda()])
    compare(got, oracle.linear_rows(x, w, s, rows), f"y > 2 GiB N={N} ctas={ctas}")
    del y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,N,path", [(256, 384, PATH_MAIN), (32, 512, PATH_DECODE)])
def test_long_k(M, N, path):
    # 40,000-byte rows: hundreds of K blocks, so every ring barrier wraps its
    # phase many times within one tile
    K = 40000
    x, w, s = synth.make_inputs(M, N, K, seed=79)
    check_full(x, w, s, Options(path=path), what=f"long K {M}x{N}x{K}")


# ------------------------------------------------------------------ concurrent host threads
def test_concurrent_host_threads_on_separate_streams():
    # The binding releases the GIL inside each C call, so these threads enter
    # the library at the same time: plan caches, the table of per-stream
    # workspaces (the K = 4127 shape repitches into its stream's) and the
    # split tail's epochs are shared.
    import threading
    cases = [
        (96, 640, 4127, None), (256, 512, 1024, None), (32, 1024, 512, Options(path=PATH_DECODE)),
        (300, 520, 640, Options(path=PATH_MAIN, mma_ctas=2, split_tail=True)),
    ]
    data = []
    for i, (M, N, K, o) in enumerate(cases):
        x, w, s = synth.make_inputs(M, N, K, seed=900 + i)
        data.append((to_dev(x), to_dev(w), to_dev(s), o, oracle.linear(x, w, s)))
    outs = [[None] * 6 for _ in cases]
    errors = []

    def worker(i):
        try:
            xd, wd, sd, o, _ = data[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for r in range(6):
                    y = torch.empty((xd.shape[0], wd.shape[0]), dtype=torch.bfloat16, device="cuda")
                    if o is None:
                        fg.fp8_gemm_scaled(xd, wd, sd, y, st)
                    else:
                        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, o, st)
                    outs[i][r] = y
            st.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    fg.check_device_error()
    for i, (_, _, _, _, ref) in enumerate(data):
        for r in range(6):
            compare(y_bits(outs[i][r]), ref, f"thread {i} call {r}")


def test_unaligned_calls_allocate_nothing_once_the_stream_has_a_workspace():
    # Calls whose rows are repitched and that bring no workspace use the one
    # the device keeps for their stream: after a stream's first such call,
    # its further calls allocate no device memory.  Two streams alternate.
    M, N, K = 320, 528, 4127
    x, w, s = synth.make_inputs(M, N, K, seed=31)
    ref = oracle.linear(x, w, s)
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    assert fg.plan(M, N, K).repitch == 1
    for i in range(2):
        fg.fp8_gemm_scaled(xd, wd, sd, ys[i], streams[i])
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for i in range(2, 8):
        fg.fp8_gemm_scaled(xd, wd, sd, ys[i], streams[i % 2])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    fg.check_device_error()
    for i, y in enumerate(ys):
        compare(y_bits(y), ref, f"stream workspace call {i}")


# ------------------------------------------------------------------ bitwise pins
@pytest.mark.parametrize("K", [4224, 4127, 1025])
def test_pair_tiles_with_odd_k_block_counts_many_calls(K):
    # With an odd number of K blocks the last stage of every tile holds one
    # K block: the odd CTA's producer of the second one has nothing to load
    # and must not wait for that stage (a stage released twice before it
    # looks is indistinguishable to a parity wait).  Hundreds of consecutive
    # calls of 2 tiles per CTA pair (33 or 9 K blocks, repitched or not)
    # must all finish without a wait running out and give identical bits.
    M, N = 2048, 4096
    x, w, s = synth.make_inputs(M, N, K, seed=K)
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    p = fg.plan(M, N, K)
    assert p.cluster == 2 and ((K + 127) // 128) % 2 == 1
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for i in range(300):
        fg.fp8_gemm_scaled(xd, wd, sd, ys[i % 3])
    fg.check_device_error()
    first = y_bits(ys[0])
    rows = np.array([0, 1, 1023, M - 1])
    compare(first[rows], oracle.linear_rows(x, w, s, rows), f"odd K blocks, K={K}")
    for y in ys[1:]:
        assert np.array_equal(y_bits(y), first)


@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
def test_one_hot_weights_reproduce_x_bitwise(path):
    M = 64 if path == PATH_DECODE else 192
    K = 256
    x, _, _ = synth.make_inputs(M, 8, K, seed=21)
    w = np.zeros((K, K), np.uint8)
    w[np.arange(K), np.arange(K)] = 0x38  # 1.0
    s = np.ones(K, np.float32)
    got = run(x, w, s, Options(path=path))
    ref = oracle.linear(x, w, s)
    g, r = oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(ref)
    assert np.array_equal(g, r)


@pytest.mark.parametrize("path_b", [PATH_MAIN, PATH_DECODE])
def test_back_to_back_calls_keep_stream_order(path_b):
    # Consecutive calls on one stream may overlap their launch and set-up
    # (programmatic dependent launch); every byte they touch must still follow
    # stream order.  Call A writes y_A; call B reads y_A's bytes as its x
    # (read after write) and writes its y over A's weight buffer (write after
    # read).  A's one-hot weight copies small integers into y_A, whose bf16
    # bytes are then all non-NaN E4M3 codes.
    ints = np.arange(-8, 9, dtype=np.float64)
    codes = synth.quantize_e4m3(ints)
    rng = np.random.default_rng(51)
    M_A = 64 if path_b == PATH_DECODE else 256
    K_A = N_A = 512
    x_a = rng.choice(codes, (M_A, K_A)).astype(np.uint8)
    w_a = np.zeros((N_A, K_A), np.uint8)
    w_a[np.arange(N_A), np.arange(K_A)] = 0x38  # 1.0
    s_a = np.ones(N_A, np.float32)
    ref_a = oracle.linear(x_a, w_a, s_a)                 # bf16 bits [M_A, N_A]
    x_b = np.ascontiguousarray(ref_a).view(np.uint8)     # [M_A, 2 N_A] bytes
    K_B, N_B = 2 * N_A, 256
    _, w_b, s_b = synth.make_inputs(M_A, N_B, K_B, seed=52)
    ref_b = oracle.linear(x_b, w_b, s_b)
    xd_a, sd_a = to_dev(x_a), to_dev(s_a)
    # A's weight buffer is big enough to hold y_B and is reused for it
    wbuf = torch.zeros(max(N_A * K_A, 2 * M_A * N_B), dtype=torch.uint8, device="cuda")
    wbuf[: N_A * K_A].copy_(torch.from_numpy(w_a.reshape(-1)))
    wd_a = wbuf[: N_A * K_A].view(N_A, K_A)
    y_a = torch.empty((M_A, N_A), dtype=torch.bfloat16, device="cuda")
    wd_b, sd_b = to_dev(w_b), to_dev(s_b)
    y_b = wbuf[: 2 * M_A * N_B].view(torch.bfloat16).view(M_A, N_B)
    for _ in range(3):
        wbuf[: N_A * K_A].copy_(torch.from_numpy(w_a.reshape(-1)))
        fg.fp8_gemm_scaled_ex(xd_a, wd_a, sd_a, y_a, Options(path=PATH_MAIN))
        fg.fp8_gemm_scaled_ex(y_a.view(torch.uint8), wd_b, sd_b, y_b, Options(path=path_b))
        fg.check_device_error()
        assert np.array_equal(y_bits(y_a), ref_a)
        compare(y_bits(y_b), ref_b, f"chained call, path {path_b}")


@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
def test_small_integer_operands_bitwise(path):
    # E4M3 codes of the integers -16..16; every partial sum stays an integer
    # below 2^24, so fp32 accumulation is exact and the only rounding is the
    # final bf16 one, which both sides take once.
    ints = np.arange(-16, 17, dtype=np.float64)
    codes = synth.quantize_e4m3(ints)
    rng = np.random.default_rng(7)
    M = 48 if path == PATH_DECODE else 160
    N, K = 272, 2048
    x = rng.choice(codes, (M, K)).astype(np.uint8)
    w = rng.choice(codes, (N, K)).astype(np.uint8)
    s = (2.0 ** -rng.integers(0, 12, N)).astype(np.float32)
    got = run(x, w, s, Options(path=path))
    ref = oracle.linear(x, w, s)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
def test_k_tail_equals_zero_padded_bitwise(path):
    M = 40 if path == PATH_DECODE else 256
    N, K, Kp = 384, 4127, 4224
    x, w, s = synth.make_inputs(M, N, K, seed=31)
    xp = np.zeros((M, Kp), np.uint8)
    wp = np.zeros((N, Kp), np.uint8)
    xp[:, :K], wp[:, :K] = x, w
    a = run(x, w, s, Options(path=path))
    b = run(xp, wp, s, Options(path=path))
    assert np.array_equal(a, b)
    compare(a, oracle.linear(x, w, s), "K=4127")


@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
def test_realign_loader_equals_tma_bitwise(path):
    M = 64 if path == PATH_DECODE else 256
    x, w, s = synth.make_inputs(M, 512, 1024, seed=41)
    a = run(x, w, s, Options(path=path))
    b = run(x, w, s, Options(path=path, force_realign=True))
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ unaligned and poisoned operands
@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
@pytest.mark.parametrize("offset", [1, 5, 15])
def test_unaligned_operand_bases_and_poisoned_neighbours(path, offset):
    """x and w start at odd byte offsets inside larger buffers whose other
    bytes are NaN codes; nothing outside [M,K] / [N,K] may leak into y."""
    M = 24 if path == PATH_DECODE else 136
    N, K = 264, 200
    x, w, s = synth.make_inputs(M, N, K, seed=offset)
    bx = torch.full((M * K + 64,), 0x7F, dtype=torch.uint8, device="cuda")
    bw = torch.full((N * K + 64,), 0xFF, dtype=torch.uint8, device="cuda")
    xd = bx[offset:offset + M * K].view(M, K)
    wd = bw[offset:offset + N * K].view(N, K)
    xd.copy_(to_dev(x))
    wd.copy_(to_dev(w))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    p = fg.plan(M, N, K, Options(path=path), x=xd, w=wd)
    assert p.repitch == 1 and p.realign == 0 and p.launches == 2
    fg.fp8_gemm_scaled_ex(xd, wd, to_dev(s), y, Options(path=path))
    fg.check_device_error()
    compare(y_bits(y), oracle.linear(x, w, s), f"offset {offset}")
    # the in-kernel loader (no workspace) gives the same bits
    y2 = torch.empty_like(y)
    fg.fp8_gemm_scaled_ex(xd, wd, to_dev(s), y2, Options(path=path, no_workspace=True))
    fg.check_device_error()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_output_guard_bands_untouched():
    M, N, K = 130, 264, 384
    x, w, s = synth.make_inputs(M, N, K, seed=3)
    for path in (PATH_MAIN, PATH_DECODE):
        Mp = M if path == PATH_MAIN else 50
        buf = torch.full((Mp * N + 2 * 512,), -12345, dtype=torch.int16, device="cuda")
        y = buf[512:512 + Mp * N].view(torch.bfloat16).view(Mp, N)
        fg.fp8_gemm_scaled_ex(to_dev(x[:Mp]), to_dev(w), to_dev(s), y, Options(path=path))
        fg.check_device_error()
        host = buf.cpu().numpy()
        assert np.all(host[:512] == -12345) and np.all(host[512 + Mp * N:] == -12345)
        compare(y_bits(y), oracle.linear(x[:Mp], w, s), f"guard path {path}")


def test_odd_n_scalar_store_path():
    # N % 8 != 0 forces the element-wise store path; y base misaligned to 2 bytes
    M, N, K = 140, 131, 256
    x, w, s = synth.make_inputs(M, N, K, seed=8)
    buf = torch.empty(M * N + 1, dtype=torch.bfloat16, device="cuda")
    y = buf[1:].view(M, N)
    fg.fp8_gemm_scaled_ex(to_dev(x), to_dev(w), to_dev(s), y, Options(path=PATH_MAIN))
    fg.check_device_error()
    compare(y_bits(y), oracle.linear(x, w, s), "odd N")


# ------------------------------------------------------------------ degenerate sizes
def test_empty_and_k_zero():
    s = to_dev(np.ones(16, np.float32))
    y = torch.full((4, 16), 7.0, dtype=torch.bfloat16, device="cuda")
    x0 = torch.empty((4, 0), dtype=torch.uint8, device="cuda")
    w0 = torch.empty((16, 0), dtype=torch.uint8, device="cuda")
    for path in (PATH_MAIN, PATH_DECODE):
        y.fill_(7.0)
        fg.fp8_gemm_scaled_ex(x0, w0, s, y, Options(path=path))
        fg.check_device_error()
        assert torch.all(y == 0)
    # M == 0: nothing launched, nothing written
    ye = torch.empty((0, 16), dtype=torch.bfloat16, device="cuda")
    fg.fp8_gemm_scaled(torch.empty((0, 8), dtype=torch.uint8, device="cuda"),
                       torch.zeros((16, 8), dtype=torch.uint8, device="cuda"), s, ye)


# ------------------------------------------------------------------ stress protocol of the pages
def test_in_place_rescale_and_same_buffer_recompute():
    """Weights and scales rescaled in place, and x overwritten in place with
    the same pointer: every call recomputes from the live contents."""
    for path, M in ((PATH_MAIN, 256), (PATH_DECODE, 32)):
        N, K = 512, 4127
        x, w, s = synth.make_inputs(M, N, K, seed=51)
        xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, Options(path=path))
        fg.check_device_error()
        compare(y_bits(y), oracle.linear(x, w, s), "first")
        s2 = (s * np.float32(3.0)).astype(np.float32)
        sd.copy_(to_dev(s2))
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, Options(path=path))
        fg.check_device_error()
        compare(y_bits(y), oracle.linear(x, w, s2), "rescaled scale")
        x2, w2, _ = synth.make_inputs(M, N, K, seed=52)
        x2[0, :] = x[0, :]  # change everything except one row
        xd.copy_(to_dev(x2))
        wd.copy_(to_dev(w2))
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, Options(path=path))
        fg.check_device_error()
        compare(y_bits(y), oracle.linear(x2, w2, s2), "new x, w in place")


# ------------------------------------------------------------------ errors and bounded waits
def test_bounded_wait_times_out_and_context_survives():
    fg.fp8_gemm_selftest_wait_timeout(2_000_000)  # 2 ms
    assert fg.fp8_gemm_check_device_error() == 5
    assert fg.lib().fp8_gemm_last_device_error_bits() & (1 << 4)
    assert fg.fp8_gemm_check_device_error() == 0  # cleared
    x, w, s = synth.workload_inputs("small")
    check_full(x, w, s, what="after timeout")


def test_rejects_host_pointers_and_aliasing():
    x = torch.zeros((4, 32), dtype=torch.uint8)
    w = torch.zeros((8, 32), dtype=torch.uint8, device="cuda")
    s = torch.ones(8, dtype=torch.float32, device="cuda")
    y = torch.empty((4, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_scaled(x, w, s, y)
    assert e.value.status == 1
    buf = torch.zeros(4 * 32 + 64, dtype=torch.uint8, device="cuda")
    xa = buf[:128].view(4, 32)
    ya = buf[64:128].view(torch.bfloat16).view(4, 8)
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_scaled(xa, w, s, ya)
    assert e.value.status == 1
    assert fg.fp8_gemm_check_device_error() == 0


def test_entry_points_leave_the_current_device_unchanged():
    """Each entry point makes the device that holds y current only for the
    call: the caller's current device is current again when it returns.  Data
    on device d is used while device (d + 1) % n is current; on a one-GPU
    machine that is the same device, and the check is that it stays current."""
    import ctypes
    lib = fg.lib()
    vp = ctypes.c_void_p
    n = torch.cuda.device_count()
    for d in range(n):
        other = (d + 1) % n
        dev = torch.device("cuda", d)
        M, N, K = 64, 256, 4127
        x, w, s = synth.make_inputs(M, N, K, 21)
        xd, wd, sd = (torch.from_numpy(a).to(dev) for a in (x, w, s))
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wp = torch.empty((N, 4128), dtype=torch.uint8, device=dev)
        xa = torch.zeros((M, 4128), dtype=torch.uint8, device=dev)
        offs = torch.tensor([0, M], dtype=torch.int32, device=dev)
        p = [vp(t.data_ptr()) for t in (xd, wd, sd, y)]
        opts = Options(mma_ctas=2, path=PATH_MAIN)._c()
        plan = fg._binding._CPlan()
        torch.cuda.set_device(other)
        calls = [
            ("scaled", lambda: lib.fp8_gemm_scaled(*p, M, N, K, None)),
            ("scaled_ex", lambda: lib.fp8_gemm_scaled_ex(*p, M, N, K, ctypes.byref(opts), None)),
            ("noalloc", lambda: lib.fp8_gemm_scaled_noalloc(*p, M, N, K, None)),
            ("prepare_weight", lambda: lib.fp8_gemm_prepare_weight(
                p[1], N, K, vp(wp.data_ptr()), 4128, None)),
            ("grouped", lambda: lib.fp8_gemm_grouped(
                vp(xa.data_ptr()), vp(wp.data_ptr()), p[2], p[3], vp(offs.data_ptr()), 1, M, N,
                4128, None, None)),
            ("plan", lambda: lib.fp8_gemm_plan(d, None, None, M, N, K, None, ctypes.byref(plan))),
        ]
        for name, call in calls:
            assert call() == 0, name
            assert torch.cuda.current_device() == other, name
        torch.cuda.set_device(d)
        assert fg.fp8_gemm_check_device_error() == 0
        # the last output written is the grouped layer's on the prepared
        # weight with zero x: every element is zero
        assert bool(torch.all(y == 0))
    torch.cuda.set_device(0)


# ------------------------------------------------------------------ CUDA graph capture
@pytest.mark.parametrize("M,N,K", [(64, 128, 256), (512, 1024, 512), (32, 2048, 1024),
                                   (300, 640, 4127), (32, 1024, 1001)])
def test_cuda_graph_capture_and_replay_with_new_data(M, N, K):
    # A captured call becomes its kernel launches (plus, when its rows must
    # be repitched, the workspace allocation and free as graph memory nodes);
    # a replay recomputes from whatever the captured buffers hold at that
    # time (nothing is cached).
    x1, w1, s1 = synth.make_inputs(M, N, K, seed=61)
    x2, w2, s2 = synth.make_inputs(M, N, K, seed=62)
    xd, wd, sd = to_dev(x1), to_dev(w1), to_dev(s1)
    x_in = to_dev(x1)  # copied into xd inside the graph: a copy node precedes the first call
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert (fg.plan(M, N, K).workspace_bytes == 0) == (K % 16 == 0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fg.fp8_gemm_scaled(xd, wd, sd, y)  # set-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        xd.copy_(x_in)
        fg.fp8_gemm_scaled(xd, wd, sd, y)
        fg.fp8_gemm_scaled(xd, wd, sd, y)  # two calls back to back in the graph
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    fg.check_device_error()
    compare(y_bits(y), oracle.linear(x1, w1, s1), "graph replay 1")
    x_in.copy_(to_dev(x2))
    wd.copy_(to_dev(w2))
    sd.copy_(to_dev(s2))
    g.replay()
    torch.cuda.synchronize()
    fg.check_device_error()
    compare(y_bits(y), oracle.linear(x2, w2, s2), "graph replay 2")


# ------------------------------------------------------------------ operand pitches, weight prepack
def pitched(a, pitch, fill=0xA5):
    """Device copy of a [rows, K] byte matrix inside a [rows, pitch] buffer
    (bytes past K poisoned), returned as the [rows, K] view."""
    rows, K = a.shape
    buf = np.full((rows, pitch), fill, np.uint8)
    buf[:, :K] = a
    return to_dev(buf)[:, :K]


@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
def test_pitched_operands_read_in_place(path):
    # pitch a multiple of 16 with K = 4127: TMA reads the operands where they
    # are (no workspace, one launch); bytes past K are never used
    M = 32 if path == PATH_DECODE else 300
    N, K, P = 520, 4127, 4144
    x, w, s = synth.make_inputs(M, N, K, seed=71)
    xv, wv = pitched(x, P), pitched(w, P)
    p = fg.plan(M, N, K, Options(path=path), x=xv, w=wv)
    assert p.workspace_bytes == 0 and p.launches == 1 and p.repitch == 0 and p.realign == 0
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fg.fp8_gemm_scaled_ex(xv, wv, to_dev(s), y, Options(path=path))
    fg.check_device_error()
    got = y_bits(y)
    compare(got, oracle.linear(x, w, s), f"pitched {path}")
    if path == PATH_MAIN:  # same K blocks and zeros as the repitched contiguous call
        assert np.array_equal(got, run(x, w, s, Options(path=path)))


@pytest.mark.parametrize("path", [PATH_MAIN, PATH_DECODE])
def test_pitched_operands_unaligned_pitch_are_repitched(path):
    M = 40 if path == PATH_DECODE else 260
    N, K, P = 300, 1000, 1013
    x, w, s = synth.make_inputs(M, N, K, seed=72)
    xv, wv = pitched(x, P), pitched(w, P)
    p = fg.plan(M, N, K, Options(path=path), x=xv, w=wv)
    assert p.repitch == 1 and p.launches == 2
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fg.fp8_gemm_scaled_ex(xv, wv, to_dev(s), y, Options(path=path))
    fg.check_device_error()
    compare(y_bits(y), oracle.linear(x, w, s), f"unaligned pitch {path}")
    # without a workspace the in-kernel loader cannot follow a pitch != K
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_scaled_ex(xv, wv, to_dev(s), y, Options(path=path, no_workspace=True))
    assert e.value.status == 2


def test_prepare_weight_leaves_only_x_to_repitch():
    M, N, K = 512, 1024, 4127
    x, w, s = synth.make_inputs(M, N, K, seed=73)
    wd = to_dev(w)
    w_out = torch.full((N, 4128), 0x5A, dtype=torch.uint8, device="cuda")
    wv = fg.fp8_gemm_prepare_weight(wd, w_out)
    torch.cuda.synchronize()
    host = w_out.cpu().numpy()
    assert np.array_equal(host[:, :K], w) and not host[:, K:].any()
    p_full = fg.plan(M, N, K, x=to_dev(x), w=wd)
    p_prep = fg.plan(M, N, K, x=to_dev(x), w=wv)
    assert p_prep.repitch == 1 and p_prep.workspace_bytes < p_full.workspace_bytes
    assert p_prep.workspace_bytes == (M * 4160 + 255) // 256 * 256  # pitch round_up(K, 64)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fg.fp8_gemm_scaled_ex(to_dev(x), wv, to_dev(s), y)
    fg.check_device_error()
    got = y_bits(y)
    assert np.array_equal(got, run(x, w, s))
    compare(got, oracle.linear(x, w, s), "prepared weight")


def test_pitch_arguments_are_checked():
    M, N, K = 64, 128, 256
    x, w, s = synth.make_inputs(M, N, K, seed=74)
    xd, wd, sd = to_dev(x), to_dev(w), to_dev(s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_scaled_ex(xd, wd, sd, y, Options(ldx=K - 1))
    assert e.value.status == 1
    out = torch.empty((N, 264), dtype=torch.uint8, device="cuda")
    with pytest.raises(fg.FP8GemmError) as e:  # ldw_out not a multiple of 16
        fg.fp8_gemm_prepare_weight(wd, out)
    assert e.value.status == 2


# ------------------------------------------------------------------ grouped (MoE) layer
def group_ranges(offs, M):
    """Row ranges the grouped layer assigns: offsets clamped to [0, M] and
    made non-decreasing (a group starts no earlier than the previous ends)."""
    clamp = lambda v: min(max(int(v), 0), M)  # noqa: E731
    ranges, prev_hi = [], 0
    for g in range(len(offs) - 1):
        lo = max(clamp(offs[g]), prev_hi)
        hi = max(clamp(offs[g + 1]), lo)
        ranges.append((lo, hi))
        prev_hi = hi
    return ranges


def run_grouped(x, w, s, offs, options=None):
    M = x.shape[0]
    G, N, _ = w.shape
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y.view(torch.int16).fill_(-1)  # sentinel: rows no group owns must keep it
    od = torch.tensor(np.asarray(offs, np.int32), device="cuda")
    fg.fp8_gemm_grouped(to_dev(x), to_dev(w), to_dev(s), y, od, options)
    fg.check_device_error()
    return y_bits(y)


@pytest.mark.parametrize("offs,M", [
    ([0, 0, 300, 317, 829, 958], 958),        # an empty group, ragged groups
    ([40, 100, 50, 2000, 20], 300),           # out of order and out of range
    ([0, 1, 2, 3, 4, 5, 6, 7, 8], 8),         # one row per group
])
def test_grouped_layer_matches_per_group_oracle(offs, M):
    G, N, K = len(offs) - 1, 384, 512
    x, _, _ = synth.make_inputs(M, 8, K, seed=81)
    rng = np.random.default_rng(82)
    w = np.stack([synth.make_inputs(8, N, K, seed=83 + g)[1] for g in range(G)])
    s = (rng.uniform(0.5, 1.5, (G, N)) / np.sqrt(K)).astype(np.float32)
    got = run_grouped(x, w, s, offs)
    covered = np.zeros(M, bool)
    for g, (lo, hi) in enumerate(group_ranges(offs, M)):
        if hi > lo:
            compare(got[lo:hi], oracle.linear(x[lo:hi], w[g], s[g]), f"group {g}")
            covered[lo:hi] = True
    assert (got[~covered] == 0xFFFF).all()


def test_grouped_layer_equals_separate_calls_on_exact_sums():
    codes = synth.quantize_e4m3(np.arange(-16, 17, dtype=np.float64))
    rng = np.random.default_rng(84)
    counts = [200, 0, 513, 64, 1]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, G, N, K = int(offs[-1]), len(counts), 256, 1024
    x = rng.choice(codes, (M, K)).astype(np.uint8)
    w = rng.choice(codes, (G, N, K)).astype(np.uint8)
    s = (2.0 ** -rng.integers(0, 12, (G, N))).astype(np.float32)
    got = run_grouped(x, w, s, offs, Options(tile_n=128))
    for g in range(G):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            assert np.array_equal(got[lo:hi], oracle.linear(x[lo:hi], w[g], s[g]))


@pytest.mark.parametrize("bn", [256, 192])
def test_grouped_layer_with_eight_epilogue_warps(bn):
    # Eight epilogue warps with a staging box per chunk: 32-row output boxes
    # that straddle a group's end are stored row by row, the others by TMA.
    offs = [0, 45, 45, 301, 333, 700, 1000]
    M, G, N, K = 1000, len(offs) - 1, 640, 256
    x, _, _ = synth.make_inputs(M, 8, K, seed=91)
    rng = np.random.default_rng(92)
    w = np.stack([synth.make_inputs(8, N, K, seed=93 + g)[1] for g in range(G)])
    s = (rng.uniform(0.5, 1.5, (G, N)) / np.sqrt(K)).astype(np.float32)
    o8 = Options(mma_ctas=2, tile_n=bn, epilogue_warps=8)
    got = run_grouped(x, w, s, offs, o8)
    for g, (lo, hi) in enumerate(group_ranges(offs, M)):
        if hi > lo:
            compare(got[lo:hi], oracle.linear(x[lo:hi], w[g], s[g]), f"group {g}, bn {bn}")
    assert np.array_equal(got, run_grouped(x, w, s, offs, Options(mma_ctas=2, tile_n=bn,
                                                                   epilogue_warps=4)))


def test_grouped_layer_argument_checks():
    M, G, N, K = 64, 2, 128, 200  # K % 16 != 0: not readable by TMA in place
    x = to_dev(np.zeros((M, K), np.uint8))
    w = to_dev(np.zeros((G, N, K), np.uint8))
    s = to_dev(np.ones((G, N), np.float32))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    od = torch.tensor([0, 32, 64], dtype=torch.int32, device="cuda")
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_grouped(x, w, s, y, od)
    assert e.value.status == 2
    with pytest.raises(fg.FP8GemmError) as e:
        fg.fp8_gemm_grouped(x[:, :192], w[:, :, :192].contiguous(), s, y, od,
                            Options(path=PATH_DECODE))
    assert e.value.status == 6
