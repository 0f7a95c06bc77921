"""Decode attention over a dense (batch, heads, length, head_dim) cache -- the pre-allocated cache
of "04 - Hacia PagedAttention (vista previa)", "Lo que funciona en la Fase 22" -- against the oracle.

The dense call reads the cache by the identity walk instead of a block table. The oracle takes a
paged pool, so each dense cache is also laid out as a pool whose block s * (S / 16) + i holds the
i-th 16 positions of sequence s, with identity tables: by "Lo que deberias llevarte de la Fase 22
sobre la Fase 27", item 2, paging changes only where rows live, so both describe the same
attention. Rows past each context are NaN-poisoned; the dense result must also equal the paged
kernel's on that pool bit for bit (same arithmetic, same split-K geometry).
"""
import ctypes

import numpy as np
import pytest

import oracle
from helpers import TOL, as_f64, to_torch
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def dense_case(dtype, lens, n_q, n_kv, d, s_max, seed, n_layers=1):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    B = len(lens)
    kd = W.normal_values(rng, (n_layers, B, n_kv, s_max, d), dtype)
    vd = W.normal_values(rng, (n_layers, B, n_kv, s_max, d), dtype)
    nanv = W.nan_value(dtype)
    for s, n in enumerate(lens):
        kd[:, s, :, n:, :] = nanv
        vd[:, s, :, n:, :] = nanv
    q = W.normal_values(rng, (B, n_q, d), dtype)
    return q, kd, vd, lens


def as_pool(dense):
    """[L, B, n_kv, S, d] -> [L, B*S/16, n_kv, 16, d]: block s*(S/16)+i = positions 16i..16i+15 of s."""
    L, B, n_kv, S, d = dense.shape
    return np.ascontiguousarray(
        dense.reshape(L, B, n_kv, S // 16, 16, d).transpose(0, 1, 3, 2, 4, 5).reshape(L, B * (S // 16), n_kv, 16, d))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d,group", [(64, 1), (128, 1), (128, 4), (256, 4), (256, 8)])
def test_dense_matches_oracle_and_paged_kernel(dtype, d, group):
    n_kv = 2
    n_q = n_kv * group
    lens = [0, 1, 15, 16, 17, 300, 1023, 1500]
    s_max = 1536
    layer = 1
    q, kd, vd, lens = dense_case(dtype, lens, n_q, n_kv, d, s_max, seed=d + group, n_layers=2)
    scale = 1.0 / np.sqrt(d)
    import torch
    desc = pkv.make_desc(dtype, 2, 1, n_q, n_kv, d)                 # num_blocks unused by the dense call
    q_t, k_t, v_t = to_torch(q, dtype), to_torch(kd, dtype), to_torch(vd, dtype)
    l_t = torch.from_numpy(lens).cuda()
    mb = s_max // 16
    ws = pkv.alloc_workspace(desc, len(lens), mb)
    out = torch.full_like(q_t, float("nan"))
    pkv.pkv_dense_decode_attention(desc, layer, q_t, k_t, v_t, l_t, scale, out, ws)
    assert pkv.pkv_get_device_status() == 0

    kp, vp = as_pool(kd), as_pool(vd)
    tables = np.arange(len(lens) * mb, dtype=np.int32).reshape(len(lens), mb)
    want = oracle.paged_decode(dtype, q, kp[layer], vp[layer], tables, lens, scale)
    got = as_f64(out)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - want)) <= TOL[dtype]
    assert np.all(got[0] == 0.0)                                         # empty context: zero row

    pdesc = pkv.make_desc(dtype, 2, kp.shape[1], n_q, n_kv, d)
    paged = torch.full_like(q_t, float("nan"))
    pkv.pkv_paged_decode_attention(pdesc, layer, q_t, to_torch(kp, dtype), to_torch(vp, dtype),
                                   torch.from_numpy(tables).cuda(), l_t, scale, paged, ws)
    assert torch.equal(paged.view(torch.uint8), out.view(torch.uint8))


def test_dense_single_partition_and_overlap_flag_bit_identical():
    """Short contexts over a grid that already fills the GPU (one partition per sequence, no
    workspace) and a launch chained to the previous one give the same bits and the oracle's values."""
    import torch
    lens = np.random.default_rng(5).integers(0, 129, size=80)
    q, kd, vd, lens = dense_case("f16", lens, 8, 8, 128, 128, seed=5)
    desc = pkv.make_desc("f16", 1, 1, 8, 8, 128)
    q_t, k_t, v_t = to_torch(q, "f16"), to_torch(kd, "f16"), to_torch(vd, "f16")
    l_t = torch.from_numpy(lens).cuda()
    per_sm, sms = pkv.pkv_decode_ctas_per_sm(desc)
    single = pkv.pkv_decode_split_geometry(desc, 80, 8, sms, per_sm)[1] == 1
    ws = pkv.alloc_workspace(desc, 80, 8)
    assert single == (ws is None)
    a = torch.empty_like(q_t)
    b = torch.empty_like(q_t)
    pkv.pkv_dense_decode_attention(desc, 0, q_t, k_t, v_t, l_t, 0.1, a, ws)
    pkv.pkv_dense_decode_attention(desc, 0, q_t, k_t, v_t, l_t, 0.1, b, ws, overlap_previous=True)
    assert torch.equal(a, b)
    tables = np.arange(80 * 8, dtype=np.int32).reshape(80, 8)
    want = oracle.paged_decode("f16", q, as_pool(kd)[0], as_pool(vd)[0], tables, lens, 0.1)
    assert np.max(np.abs(as_f64(a) - want)) <= TOL["f16"]
    assert pkv.pkv_get_device_status() == 0


def test_dense_rejects_bad_lengths_before_launch():
    import torch
    desc = pkv.make_desc("f16", 1, 1, 4, 4, 64)
    q = torch.zeros((2, 4, 64), dtype=torch.float16, device="cuda")
    cache = torch.zeros((1, 2, 4, 32, 64), dtype=torch.float16, device="cuda")
    lens = torch.tensor([3, 20], dtype=torch.int32, device="cuda")
    L = pkv.lib()
    vp = ctypes.c_void_p
    before = pkv.pkv_launch_count()
    for s_max in (0, 24, -16):                                           # not a positive multiple of 16
        rc = L.pkv_dense_decode_attention(ctypes.byref(desc), 0, vp(q.data_ptr()), vp(cache.data_ptr()),
                                          vp(cache.data_ptr()), s_max, vp(lens.data_ptr()), 2, ctypes.c_float(1.0),
                                          vp(q.data_ptr()), vp(0), 0, 0, vp(0))
        assert rc == pkv.PKV_ERR_INVALID_ARG
    rc = L.pkv_dense_decode_attention(ctypes.byref(desc), 0, vp(q.data_ptr()), vp(cache.data_ptr()),
                                      vp(cache.data_ptr()), 32, vp(lens.data_ptr()), 2, ctypes.c_float(1.0),
                                      vp(q.data_ptr()), vp(0), 0, 2, vp(0))  # unknown flag bit
    assert rc == pkv.PKV_ERR_INVALID_ARG
    assert pkv.pkv_launch_count() == before


def test_dense_fullsize_gpt_layer_sampled():
    """The dense comparison at the GPT-style batch's full size (64 sequences x 32 heads x 128 fp16,
    lengths of the bench's workload, one layer), as bench.py times it: sampled sequences against
    the oracle on their rows laid out as a pool with identity tables."""
    import torch
    wl = W.gpt(seed=W.BASE_SEED + 1)
    L, B, n_kv, d = 1, wl.n_seqs, wl.n_kv_heads, wl.head_dim
    lens = wl.context_lens.astype(np.int32)
    s_max = int(-(-int(lens.max()) // 16) * 16)
    desc = pkv.make_desc("f16", L, 1, wl.n_q_heads, n_kv, d)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    shape = pkv.dense_cache_shape(desc, B, s_max)
    kc = torch.randn(shape, dtype=torch.float16, device="cuda", generator=g)
    vc = torch.randn(shape, dtype=torch.float16, device="cuda", generator=g)
    for s in range(B):                                   # rows past each context: never read
        kc[:, s, :, int(lens[s]):] = float("nan")
        vc[:, s, :, int(lens[s]):] = float("nan")
    q = torch.randn((B, wl.n_q_heads, d), dtype=torch.float16, device="cuda", generator=g)
    out = torch.full_like(q, float("nan"))
    l_t = torch.from_numpy(lens).cuda()
    ws = pkv.alloc_workspace(desc, B, s_max // 16)
    pkv.pkv_dense_decode_attention(desc, 0, q, kc, vc, l_t, wl.scale, out, ws)
    assert pkv.pkv_get_device_status() == 0
    assert torch.isfinite(out.float()).all()
    sel = [0, 9, 31, int(np.argmax(lens)), 63]
    for s in sel:
        kd = kc[:, s:s + 1].cpu().numpy()
        vd = vc[:, s:s + 1].cpu().numpy()
        tables = np.arange(s_max // 16, dtype=np.int32).reshape(1, -1)
        want = oracle.paged_decode("f16", q[s:s + 1].cpu().numpy(), as_pool(kd)[0], as_pool(vd)[0], tables,
                                   lens[s:s + 1], wl.scale)
        assert np.max(np.abs(as_f64(out[s:s + 1]) - want)) <= TOL["f16"], s
