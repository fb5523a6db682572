"""The planner on the host, for a described GB300 (152 SMs, 227 KB opt-in shared memory,
compute capability 10.3) and for devices without the tensor-core family: every plan the
library would launch stays inside the hardware limits, only wgrad asks for memory beyond its
arguments (the caller's workspace), the tensor-core forward splits K only when its column
tiles fill fewer than half the SMs and then into one thread-block cluster of at most 8 CTAs
per tile, and forcing a family is honoured.  No GPU: conv_query_for_device makes no CUDA
call."""
import pytest

from implicit_gemm_conv2d_gb300 import binding

GB300 = binding.GB300
MAX_CLUSTER = 8
OPS = (binding.OP_FWD, binding.OP_BWD_DATA, binding.OP_BWD_FILTER, binding.OP_BWD_BIAS, binding.OP_FWD_WS,
       binding.OP_BWD_DATA_WS, binding.OP_BWD)
WS_OPS = (binding.OP_BWD_FILTER, binding.OP_FWD_WS, binding.OP_BWD_DATA_WS, binding.OP_BWD)

SHAPES = {
    "L1": (59, 128, 11, 15, 5, 3, 1),
    "L2": (128, 128, 3, 4, 3, 1, 0),
    "odd": (3, 5, 7, 9, 2, 2, 1),
    "wide_oc_p16": (4, 200, 6, 6, 3, 1, 0),
    "kk_above_128": (2, 8, 13, 12, 12, 1, 1),
    "k1": (16, 24, 3, 5, 1, 1, 0),
    "k_eq_input": (7, 33, 5, 5, 5, 2, 1),
    "stride_gt_k": (5, 20, 10, 11, 2, 3, 0),
    "long_rows": (1, 3, 120, 120, 1, 1, 0),
    "k1_wide": (160, 64, 4, 5, 1, 1, 1),
}
BATCHES = (1, 37, 256, 1024, 4096, 16384, 32768)


@pytest.fixture(autouse=True)
def _restore_algo():
    yield
    for op in OPS:
        if op != binding.OP_BWD:  # set through d_input's and wgrad's choices
            binding.conv_set_algo(op, binding.ALGO_AUTO)


def plan(op, B, shape, dtype, dev=GB300):
    IC, OC, H, W, K, S, relu = shape
    return binding.conv_query_for_device(op, binding.make_desc(B, IC, OC, H, W, K, S, relu, dtype), **dev)


@pytest.mark.parametrize("dtype", [binding.F32, binding.BF16])
@pytest.mark.parametrize("name", list(SHAPES))
def test_plans_within_limits(name, dtype):
    IC, OC, H, W, K, S, relu = SHAPES[name]
    OH, OW = (H - K) // S + 1, (W - K) // S + 1
    for B in BATCHES:
        if B * IC * H * W >= 2 ** 31:
            continue
        for op in OPS:
            q = plan(op, B, SHAPES[name], dtype)
            where = (name, dtype, B, op, q)
            assert q["launches"] >= 1, where
            assert 32 <= q["block"] <= 1024 and q["block"] % 32 == 0, where
            assert 0 <= q["smem_bytes"] <= GB300["smem_optin"], where
            assert q["grid"] >= 1, where
            if q["algo"] == binding.ALGO_TC and op != binding.OP_BWD:
                assert q["grid"] <= GB300["sms"], where  # persistent (the fused backward adds one CTA per wgrad tile)
            if op == binding.OP_BWD and q["algo"] == binding.ALGO_TC:
                assert q["launches"] == 3 and q["workspace"] > 0 and q["splits"] >= 1, where
            if op not in WS_OPS:
                assert q["workspace"] == 0, where
            if op in (binding.OP_FWD_WS, binding.OP_BWD_DATA_WS):
                # the workspace path packs the weights into the workspace, then the main kernel
                if q["algo"] == binding.ALGO_TC:
                    assert q["launches"] == 2 and q["workspace"] > 0, where
                else:
                    assert q["workspace"] == 0, where
            if op == binding.OP_FWD and q["algo"] == binding.ALGO_TC:
                # one launch: weights formatted in the kernel, K ranges reduced in a cluster
                assert q["launches"] == 1 and 1 <= q["splits"] <= MAX_CLUSTER, where
                if q["splits"] > 1:
                    assert q["grid"] % q["splits"] == 0, where
            if op == binding.OP_BWD_DATA and q["algo"] == binding.ALGO_TC:
                assert q["launches"] == 1, where
            if op == binding.OP_BWD_FILTER and q["splits"] > 0:
                assert q["workspace"] >= q["splits"] * OC * IC * K * K * 4, where
            if op == binding.OP_BWD_BIAS:
                if q["algo"] == binding.ALGO_FFMA:
                    assert 256 <= q["block"] <= 1024 and q["smem_bytes"] <= 48 * 1024, where
                    assert q["splits"] in (1, 2, 4, 8) and q["grid"] % q["splits"] == 0, where
                    assert q["launches"] == 1, where
                else:
                    assert q["algo"] == binding.ALGO_DIRECT and OH * OW > 12288, where


def test_bias_gradient_threads_grow_with_rows_per_range():
    # 256 threads while the sample ranges are short (B = 1024: 8 ranges of 128 rows), up to
    # 1024 threads (about 8 rows per row lane) at the PR's bias-gradient batch
    for name in ("L1", "L2"):
        for dtype in (binding.F32, binding.BF16):
            assert plan(binding.OP_BWD_BIAS, 1024, SHAPES[name], dtype)["block"] == 256
            assert plan(binding.OP_BWD_BIAS, 32768, SHAPES[name], dtype)["block"] == 1024


def test_encoder_layers_use_tensor_cores_on_gb300():
    for name in ("L1", "L2"):
        for dtype in (binding.F32, binding.BF16):
            for op in (binding.OP_FWD, binding.OP_BWD_DATA, binding.OP_BWD_FILTER):
                assert plan(op, 1024, SHAPES[name], dtype)["algo"] == binding.ALGO_TC, (name, dtype, op)


@pytest.mark.parametrize("dtype", [binding.F32, binding.BF16])
def test_forward_k_ranges_only_with_few_column_tiles(dtype):
    # layer 1 at B = 1024: 12288 columns = 96 tiles of 128, more than half of 152 SMs
    q = plan(binding.OP_FWD, 1024, SHAPES["L1"], dtype)
    assert q["splits"] == 1 and q["grid"] == 96
    # layer 2 at B = 1024: 2048 columns = 16 tiles: K splits into a cluster of ranges per
    # tile, one CTA per (tile, range), and the work items fill at least half the SMs
    q = plan(binding.OP_FWD, 1024, SHAPES["L2"], dtype)
    assert 1 < q["splits"] <= MAX_CLUSTER and q["grid"] == 16 * q["splits"] >= GB300["sms"] // 2
    # large batches never split
    for name in ("L1", "L2"):
        assert plan(binding.OP_FWD, 16384, SHAPES[name], dtype)["splits"] == 1


def test_no_tensor_core_plan_without_the_hardware():
    hopper = dict(sms=132, smem_optin=232448, cc_major=9, cc_minor=0)
    small = dict(sms=152, smem_optin=48 * 1024, cc_major=10, cc_minor=3)
    for op in (binding.OP_FWD, binding.OP_BWD_DATA, binding.OP_BWD_FILTER):
        for name in SHAPES:
            q = plan(op, 1024, SHAPES[name], binding.F32, hopper)
            assert q["algo"] in (binding.ALGO_FFMA, binding.ALGO_DIRECT), (op, name, q)
            q = plan(op, 1024, SHAPES[name], binding.F32, small)
            assert q["smem_bytes"] <= small["smem_optin"], (op, name, q)
            if name in ("L1", "L2"):  # their tensor-core stages need more than 48 KB
                assert q["algo"] != binding.ALGO_TC, (op, name, q)


def test_backward_fused_only_below_two_waves_of_d_input_items():
    # layer 1: d_input has one sample tile of 10 samples per work item, 152 SMs: fused below
    # 3040 samples, two calls from there on; layer 2 (64 samples per tile) fuses to 16384
    for dtype in (binding.F32, binding.BF16):
        for B, want in ((1, binding.ALGO_TC), (1024, binding.ALGO_TC), (3000, binding.ALGO_TC),
                        (4096, binding.ALGO_AUTO), (16384, binding.ALGO_AUTO)):
            q = plan(binding.OP_BWD, B, SHAPES["L1"], dtype)
            assert q["algo"] == want, (dtype, B, q)
        for B, want in ((1024, binding.ALGO_TC), (16384, binding.ALGO_TC), (32768, binding.ALGO_AUTO)):
            assert plan(binding.OP_BWD, B, SHAPES["L2"], dtype)["algo"] == want, (dtype, B)
        # fused: the wgrad tiles fill about two thirds of the SMs
        q = plan(binding.OP_BWD, 1024, SHAPES["L1"], dtype)
        w = plan(binding.OP_BWD_FILTER, 1024, SHAPES["L1"], dtype)
        tiles = w["grid"] // w["splits"]
        assert abs(tiles * q["splits"] - 2 * GB300["sms"] // 3) <= tiles // 2 + 1, (q, w)
        # two calls: the workspace holds both operations' parts
        q = plan(binding.OP_BWD, 16384, SHAPES["L1"], dtype)
        a = plan(binding.OP_BWD_DATA_WS, 16384, SHAPES["L1"], dtype)
        w = plan(binding.OP_BWD_FILTER, 16384, SHAPES["L1"], dtype)
        assert q["workspace"] >= a["workspace"] + w["workspace"] and q["splits"] == w["splits"], (q, a, w)


def test_workspace_path_matches_the_plain_plan():
    # the same family (the packed stages need no raw w slots, so the workspace path may pick a
    # deeper ring), with a workspace for the packed image
    for name in ("L1", "L2"):
        for dtype in (binding.F32, binding.BF16):
            for B in (37, 1024, 16384):
                for plain_op, ws_op in ((binding.OP_FWD, binding.OP_FWD_WS), (binding.OP_BWD_DATA, binding.OP_BWD_DATA_WS)):
                    a, b = plan(plain_op, B, SHAPES[name], dtype), plan(ws_op, B, SHAPES[name], dtype)
                    assert a["algo"] == b["algo"] == binding.ALGO_TC, (name, dtype, B, a, b)
                    assert b["workspace"] > 0 and a["workspace"] == 0, (name, dtype, B, a, b)


def test_forced_family_is_honoured():
    for op in OPS:
        if op == binding.OP_BWD:
            continue  # set through its two operations
        binding.conv_set_algo(op, binding.ALGO_DIRECT)
        assert plan(op, 1024, SHAPES["L1"], binding.F32)["algo"] == binding.ALGO_DIRECT
        binding.conv_set_algo(op, binding.ALGO_AUTO)
    binding.conv_set_algo(binding.OP_BWD_DATA, binding.ALGO_FFMA)
    assert plan(binding.OP_BWD, 1024, SHAPES["L1"], binding.F32)["algo"] == binding.ALGO_AUTO  # two calls
    binding.conv_set_algo(binding.OP_BWD_DATA, binding.ALGO_AUTO)
    assert plan(binding.OP_BWD, 1024, SHAPES["L1"], binding.F32)["algo"] == binding.ALGO_TC
    binding.conv_set_algo(binding.OP_FWD, binding.ALGO_TC)
    with pytest.raises(binding.ConvError):  # no tensor cores on this device: the forced family cannot run
        plan(binding.OP_FWD, 1024, SHAPES["L1"], binding.F32, dict(sms=132, smem_optin=232448, cc_major=9,
                                                                   cc_minor=0))


def test_device_properties_checked():
    d = binding.make_desc(8, 59, 128, 11, 15, 5, 3, 1, binding.F32)
    for bad in (dict(GB300, sms=0), dict(GB300, smem_optin=0), dict(GB300, cc_major=0), dict(GB300, cc_minor=-1)):
        with pytest.raises(binding.ConvError):
            binding.conv_query_for_device(binding.OP_FWD, d, **bad)


def test_wgrad_k_tile_rows_per_dtype_and_batch():
    # fp32 and small-batch bf16 keep the patches in tensor memory (k-tiles of 128 rows, the TMEM
    # lanes); bf16 from 2048 samples keeps g there instead and takes k-tiles of 256 rows
    for name in ("L1", "L2"):
        IC, OC, H, W, K, S, relu = SHAPES[name]
        kred = IC * K * K
        for dtype in (binding.F32, binding.BF16):
            for B in (37, 1024, 2047, 2048, 4096, 16384):
                w = plan(binding.OP_BWD_FILTER, B, SHAPES[name], dtype)
                rows = 256 if (dtype == binding.BF16 and B >= 2048) else 128
                want = -(-kred // min(rows, -(-kred // 32) * 32)) * -(-OC // 128)
                assert w["algo"] == binding.ALGO_TC and w["grid"] == want * w["splits"], (name, dtype, B, w)
