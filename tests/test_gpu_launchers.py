"""The per-step launchers (pkv.decode_append_launcher, prefill_launcher, append_launcher).

They check a step's [L, ...] tensors once and then launch each layer with one C call; a layer's
results must be bit-identical to the per-call bindings on the same inputs (also when the tensors
are views of larger buffers), and the checks must refuse what the per-call bindings refuse.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W
from paged_kv_cache_258_gb300.engine import PagedKVCache

pytestmark = pytest.mark.gpu

L, NQ, NKV, D, NB, MB = 3, 8, 2, 128, 96, 16


def _cache(dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    desc = pkv.make_desc(dtype, L, NB, NQ, NKV, D)
    cache = PagedKVCache(desc, free_order=W.free_order(NB, seed))
    cache.k_pool.normal_(generator=g)
    cache.v_pool.normal_(generator=g)
    return desc, cache, g


def _rows(g, shape, dtype, big=None):
    """[L, n, ...] rows; with big, a view [:, :n] of a larger [L, big, ...] buffer."""
    dt = pkv.torch_dtype(dtype)
    if big is None:
        return torch.randn(shape, generator=g, device="cuda").to(dt)
    full = torch.randn((shape[0], big) + tuple(shape[2:]), generator=g, device="cuda").to(dt)
    return full[:, : shape[1]]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("view", [False, True])
def test_decode_launcher_matches_per_call_binding(dtype, view):
    desc, cache, g = _cache(dtype, 11)
    lens0 = [17, 40, 1, 33, 64]
    n = len(lens0)
    for s, c in enumerate(lens0):
        assert cache.mgr.add_seq(s, c)[0] == pkv.PKV_OK
    for s in range(n):
        assert cache.mgr.append_slot(s)[0] == pkv.PKV_OK  # the step's new row at position len - 1
    rc, tables, lens = cache.mgr.pack_tables(list(range(n)), MB)
    assert rc == pkv.PKV_OK
    tables, lens = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    q = _rows(g, (L, n, NQ, D), dtype, 9 if view else None)
    k = _rows(g, (L, n, NKV, D), dtype, 9 if view else None)
    v = _rows(g, (L, n, NKV, D), dtype, 9 if view else None)
    ws = pkv.alloc_workspace(desc, n, MB)
    out_a = torch.full((L, n, NQ, D), float("nan"), device="cuda").to(q.dtype)
    out_b = out_a.clone()
    pools0 = (cache.k_pool.clone(), cache.v_pool.clone())
    for layer in range(L):
        pkv.pkv_paged_decode_append_attention(desc, layer, q[layer], k[layer], v[layer], cache.k_pool,
                                              cache.v_pool, tables, lens, 0.09, out_a[layer], ws)
    pools_a = (cache.k_pool.clone(), cache.v_pool.clone())
    cache.k_pool.copy_(pools0[0])
    cache.v_pool.copy_(pools0[1])
    launch = pkv.decode_append_launcher(desc, q, k, v, cache.k_pool, cache.v_pool, tables, lens, 0.09, out_b, ws)
    for layer in range(L):
        launch(layer, layer > 0)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_status() == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(pools_a[0].view(torch.int16), cache.k_pool.view(torch.int16))
    assert torch.equal(pools_a[1].view(torch.int16), cache.v_pool.view(torch.int16))


@pytest.mark.parametrize("view", [False, True])
def test_prefill_and_append_launchers_match_per_call_bindings(view):
    dtype = "bf16"
    desc, cache, g = _cache(dtype, 12)
    chunks = [(0, 70), (1, 33), (2, 129)]
    n_tok = sum(c for _, c in chunks)
    slots = []
    for sid, c in chunks:
        rc, sl = cache.mgr.add_seq(sid, c)
        assert rc == pkv.PKV_OK
        slots.append(sl)
    slots = torch.from_numpy(np.concatenate(slots)).cuda()
    rc, tables, lens = cache.mgr.pack_tables([sid for sid, _ in chunks], MB)
    assert rc == pkv.PKV_OK
    tables, lens = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    qs = torch.tensor(np.concatenate([[0], np.cumsum([c for _, c in chunks])]), dtype=torch.int32).cuda()
    q = _rows(g, (L, n_tok, NQ, D), dtype, n_tok + 7 if view else None)
    k = _rows(g, (L, n_tok, NKV, D), dtype, n_tok + 7 if view else None)
    v = _rows(g, (L, n_tok, NKV, D), dtype, n_tok + 7 if view else None)
    max_q = max(c for _, c in chunks)
    out_a = torch.zeros((L, n_tok, NQ, D), device="cuda").to(q.dtype)
    out_b = out_a.clone()
    pools0 = (cache.k_pool.clone(), cache.v_pool.clone())
    for layer in range(L):
        pkv.pkv_kv_append(desc, layer, k[layer], v[layer], slots, cache.k_pool, cache.v_pool)
        pkv.pkv_paged_prefill_attention(desc, layer, q[layer], cache.k_pool, cache.v_pool, tables, lens, qs, max_q,
                                        0.07, out_a[layer])
    pools_a = (cache.k_pool.clone(), cache.v_pool.clone())
    cache.k_pool.copy_(pools0[0])
    cache.v_pool.copy_(pools0[1])
    append = pkv.append_launcher(desc, k, v, slots, cache.k_pool, cache.v_pool)
    attend = pkv.prefill_launcher(desc, q, cache.k_pool, cache.v_pool, tables, lens, qs, max_q, 0.07, out_b)
    for layer in range(L):
        append(layer)
    for layer in range(L):
        attend(layer, layer > 0)
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_status() == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(pools_a[0].view(torch.int16), cache.k_pool.view(torch.int16))
    assert torch.equal(pools_a[1].view(torch.int16), cache.v_pool.view(torch.int16))


def test_launchers_refuse_bad_tensors():
    desc, cache, g = _cache("f16", 13)
    n = 2
    q = _rows(g, (L, n, NQ, D), "f16")
    k = _rows(g, (L, n, NKV, D), "f16")
    tables = torch.zeros((n, MB), dtype=torch.int32, device="cuda")
    lens = torch.ones(n, dtype=torch.int32, device="cuda")
    ws = pkv.alloc_workspace(desc, n, MB)

    def dec(**kw):
        args = dict(q=q, k_new=k, v_new=k, k_pool=cache.k_pool, v_pool=cache.v_pool, block_tables=tables,
                    context_lens=lens, scale=0.1, out=q.clone(), workspace=ws)
        args.update(kw)
        return pkv.decode_append_launcher(desc, **args)

    dec()  # the unmodified arguments are accepted
    with pytest.raises(ValueError):
        dec(q=q.float())                                     # dtype
    with pytest.raises(ValueError):
        dec(q=q[:2])                                         # not every layer
    with pytest.raises(ValueError):
        dec(q=q.transpose(2, 3).contiguous().transpose(2, 3))  # a layer's slice is not contiguous
    with pytest.raises(ValueError):
        dec(out=q.cpu())                                     # host memory
    with pytest.raises(ValueError):
        dec(block_tables=tables[:1])                         # tables of another batch size
    with pytest.raises(ValueError):
        pkv.append_launcher(desc, k, k.to(torch.bfloat16), torch.zeros(n, dtype=torch.int64, device="cuda"),
                            cache.k_pool, cache.v_pool)
    with pytest.raises(ValueError):
        pkv.prefill_launcher(desc, q, cache.k_pool, cache.v_pool, tables, lens,
                             torch.zeros(n, dtype=torch.int32, device="cuda"), 1, 0.1, q.clone())  # query_start size
