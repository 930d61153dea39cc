"""NVFP4 append through the C ABI vs the oracle: the whole cache bit-exact
(untouched bytes keep the 0xA5 sentinel), device-checked scales, no host sync.

The failure cases follow the FlashInfer PR #6204 analysis page ("NVFP4 KV 캐시
어펜드 성능 최적화로 인한 동기화 제거", test section): a bad CUDA scale must
surface from the kernel in eager and graph mode.  Here the kernel reports it
through the status word instead of trapping, and the context stays usable.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import cache_to_host, device_inputs, fi, gpu_cache, oracle_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _assert_cache_equal(gpu_c, host_c):
    g = cache_to_host(gpu_c)
    for name in ("k_data", "v_data", "k_sf", "v_sf"):
        diff = np.argwhere(g[name] != host_c[name])
        assert diff.size == 0, f"{name}: {len(diff)} bytes differ, first at {diff[:4].tolist()}"


@pytest.mark.parametrize("name", ["tiny", "append", "ragged_small", "ragged_small_d64", "mha_small_d64",
                                  "decode_ps128"])
@pytest.mark.parametrize("host_scale", [False, True])
def test_append_bit_exact(name, host_scale):
    m = fi()
    d = device_inputs(name)
    c = gpu_cache(d)
    ctx = m.fi_context_create()
    if host_scale:
        m.fi_nvfp4_append_host_scale(ctx, d["k"], d["v"], d["k_scale"], d["v_scale"],
                                     d["slot_mapping"], c)
    else:
        m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    _assert_cache_equal(c, oracle_cache(d))


def test_append_strided_rows_and_edge_blocks(oracle):
    """Token stride larger than H*D (rows of a fused QKV buffer), blocks that
    are all zero, all -0, tiny (s8 underflow), huge (saturation)."""
    m = fi()
    N, H, D, ps, P = 70, 2, 128, 16, 6
    g = torch.Generator().manual_seed(1)
    base = torch.randn((N, 3 * H * D), generator=g)
    base[0, :16] = 0.0
    base[1, :16] = -0.0
    base[2, :16] = 1e-30
    base[3, :16] = 3e4
    base[4, 16:32] = torch.tensor([2688.0, -2688, 224, 112, 0, -0.0, 336, 560, 672, 784,
                                   1120, 1344, 1568, 2240, -1344, 100])
    buf = base.to(torch.bfloat16).cuda()
    k = buf[:, :H * D].view(N, H, D)
    v = buf[:, H * D:2 * H * D].view(N, H, D)
    slots = torch.randperm(P * ps, generator=g)[:N].to(torch.int64)
    slots[5] = -1
    c = m.NVFP4Cache(P, H, ps, D, fill=0xA5)
    c.k_scale.fill_(1.0)
    c.v_scale.fill_(0.003)
    ctx = m.fi_context_create()
    m.fi_nvfp4_append(ctx, k, v, c.k_scale, c.v_scale, slots.cuda(), c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    host = oracle.new_cache(P, H, ps, D)
    kb = W.bits(buf[:, :H * D].reshape(N, H, D))
    vb = W.bits(buf[:, H * D:2 * H * D].reshape(N, H, D))
    assert oracle.append(kb, vb, 1.0, 0.003, slots.numpy(), host) == 0
    _assert_cache_equal(c, host)


@pytest.mark.parametrize("H,D,N,gk,gv", [
    (72, 128, 37, 1.0, 0.003),          # rows of 9216 elements: the direct kernel
    (160, 64, 20, 0.5, 2.0),            # the same at D = 64
    (8, 128, 333, 1e-32, 7e30),         # staged; RN(6 g) outside the Markstein range
    (2, 64, 1000, 1e-39, 3e-5),         # staged, 32 tokens per stage; subnormal g
])
def test_append_wide_rows_ragged_stages_extreme_scales(oracle, H, D, N, gk, gv):
    """Both append kernels (rows that fit a shared-memory stage and rows that
    do not), a partial last stage, blocks whose amax is below 2^-100 or far
    above 1, and global scales on both sides of the fast division's range:
    the whole cache must equal the oracle's bytes."""
    m = fi()
    ps = 16
    P = (N + ps - 1) // ps + 3
    g = torch.Generator().manual_seed(H * 1000 + N)
    x = torch.randn((2, N, H, D), generator=g)
    mag = torch.tensor([1.0, 1e-33, 1e-20, 1e4, 1e30, 3e-5])
    pick = torch.randint(0, len(mag), (2, N, H, D // 16, 1), generator=g)
    x = (x.view(2, N, H, D // 16, 16) * mag[pick]).view(2, N, H, D)
    kv = x.to(torch.bfloat16)
    slots = torch.randperm(P * ps, generator=g)[:N].to(torch.int64)
    slots[:: 7] = -1
    c = m.NVFP4Cache(P, H, ps, D, fill=0xA5)
    c.k_scale.fill_(gk)
    c.v_scale.fill_(gv)
    ctx = m.fi_context_create()
    m.fi_nvfp4_append(ctx, kv[0].cuda(), kv[1].cuda(), c.k_scale, c.v_scale, slots.cuda(), c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    host = oracle.new_cache(P, H, ps, D)
    sk = float(np.float32(gk))
    sv = float(np.float32(gv))
    assert oracle.append(W.bits(kv[0]), W.bits(kv[1]), sk, sv, slots.numpy(), host) == 0
    _assert_cache_equal(c, host)


@pytest.mark.parametrize("H,D,N,strided", [
    (8, 128, 70001, False),   # dense token rows: one bulk copy per tensor and stage
    (4, 64, 66000, True),     # rows of a wider buffer: one bulk copy per token row
])
def test_append_long_staged(oracle, H, D, N, strided):
    """Appends of 65536 tokens or more take the shared-memory staged kernel:
    whole cache bit-exact against the oracle, with a partial last stage,
    skipped and repeated-page slots."""
    m = fi()
    ps = 16
    P = (N + ps - 1) // ps + 5
    g = torch.Generator().manual_seed(N)
    width = 3 * H * D if strided else H * D
    base = torch.randn((N, 2 * width), generator=g).to(torch.bfloat16)
    k = base[:, :H * D].view(N, H, D)
    v = base[:, width:width + H * D].view(N, H, D)
    slots = torch.randperm(P * ps, generator=g)[:N].to(torch.int64)
    slots[::13] = -1
    c = m.NVFP4Cache(P, H, ps, D, fill=0xA5)
    c.k_scale.fill_(0.0021)
    c.v_scale.fill_(0.0017)
    bd = base.cuda()
    kd = bd[:, :H * D].view(N, H, D)
    vd = bd[:, width:width + H * D].view(N, H, D)
    ctx = m.fi_context_create()
    m.fi_nvfp4_append(ctx, kd, vd, c.k_scale, c.v_scale, slots.cuda(), c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    host = oracle.new_cache(P, H, ps, D)
    sk = float(np.float32(0.0021))
    sv = float(np.float32(0.0017))
    assert oracle.append(W.bits(k.contiguous()), W.bits(v.contiguous()), sk, sv, slots.numpy(),
                         host) == 0
    _assert_cache_equal(c, host)


@pytest.mark.parametrize("mode", ["eager", "graph"])
@pytest.mark.parametrize("bad", [0.0, -0.0, -1.0, float("inf"), float("nan")])
def test_bad_device_scale_sets_flag_and_writes_nothing(mode, bad):
    m = fi()
    d = device_inputs("tiny")
    c = gpu_cache(d)
    ctx = m.fi_context_create()
    c.v_scale.fill_(bad)
    if mode == "eager":
        m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    else:
        s = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c,
                                  stream=s)
        graph.replay()
    bits = m.fi_device_status(ctx)
    assert bits == m.FI_DEV_BAD_V_SCALE
    for t in (c.k_data, c.v_data, c.k_sf, c.v_sf):
        assert bool((t == 0xA5).all())
    # the context is still usable: a good append afterwards is bit-exact
    c.v_scale.fill_(d["v_scale"])
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    _assert_cache_equal(c, oracle_cache(d))


def test_host_scale_rejected_on_host():
    m = fi()
    d = device_inputs("tiny")
    c = gpu_cache(d)
    ctx = m.fi_context_create()
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(m.FiError) as e:
            m.fi_nvfp4_append_host_scale(ctx, d["k"], d["v"], bad, 0.1, d["slot_mapping"], c)
        assert e.value.status == m.FI_ERR_BAD_SCALE
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)


def test_empty_append_checks_nothing():
    m = fi()
    d = device_inputs("tiny")
    c = gpu_cache(d)
    c.k_scale.fill_(float("nan"))
    ctx = m.fi_context_create()
    m.fi_nvfp4_append(ctx, d["k"][:0], d["v"][:0], c.k_scale, c.v_scale, d["slot_mapping"][:0], c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)


def test_slot_out_of_range_flagged():
    m = fi()
    d = device_inputs("tiny")
    c = gpu_cache(d)
    slots = d["slot_mapping"].clone()
    slots[3] = c.num_pages * c.page_size + 5
    ctx = m.fi_context_create()
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, slots, c)
    assert m.fi_device_status(ctx) == m.FI_DEV_SLOT_OOB
    m.fi_context_destroy(ctx)
    mask = torch.ones(slots.numel(), dtype=torch.bool)
    mask[3] = False
    _assert_cache_equal(c, oracle_cache(d, token_mask=mask))


def test_append_captures_in_graph_and_does_not_sync():
    """Capture must succeed (any host read of device memory would break it)
    and replay must equal the eager result."""
    m = fi()
    d = device_inputs("append")
    c = gpu_cache(d)
    ctx = m.fi_context_create()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c,
                              stream=s)
    graph.replay()
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    _assert_cache_equal(c, oracle_cache(d))
