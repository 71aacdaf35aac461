"""CPU-only checks of the boundary and host logic: the library loads and
exports every entry point the header declares, the paged allocator follows
its rules, and replica aggregation works across two gloo ranks."""
import os
import re
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from lossless_speculative_decoding_gb300 import build, binding
    build.build()
    return binding


def test_exports_match_header(B):
    hdr = open(os.path.join(ROOT, "include", "spec.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    declared = set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", hdr))
    lib = B.lib()
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(B.EXPORTS)


def test_strerror(B):
    assert B.spec_strerror(-2) == "KV page pool exhausted"
    assert B.spec_strerror(0) == "ok"


def test_tensor_sizes_match_generator(B):
    import synthetic as syn
    for cfg in (syn.TINY, syn.MOE3B, syn.MOE3B_FP8, syn.DENSE4B):
        c = B.make_config(n_layers=cfg.n_layers, hidden=cfg.hidden, n_q_heads=cfg.n_q_heads,
                          n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, n_experts=cfg.n_experts,
                          top_k=cfg.top_k, n_shared=cfg.n_shared, inter=cfg.inter, vocab=cfg.vocab,
                          wdtype=cfg.wdtype)
        specs = syn.tensor_specs(cfg)
        assert B.spec_tensor_count(c) == len(specs)
        size = {syn.F32: 4, syn.BF16: 2, syn.FP8: 1}
        for i, (_, shape, dt, _) in enumerate(specs):
            assert B.spec_tensor_bytes(c, i) == int(np.prod(shape)) * size[dt], (cfg.name, i)


def test_pool_reserve_commit_release(B):
    p = B.spec_pool_create(10, 16, 3, 8)
    assert B.spec_pool_reserve(p, 0, 33) == 0                  # 3 pages
    assert B.spec_pool_block_table(p, 0) == [0, 1, 2]
    assert B.spec_pool_free_count(p) == 7
    assert B.spec_pool_commit(p, 0, 17, 0) == 0                # keeps ceil(17/16) = 2 pages
    assert B.spec_pool_block_table(p, 0) == [0, 1]
    assert B.spec_pool_free_count(p) == 8
    assert B.spec_pool_reserve(p, 0, 16 * 9) == -1             # beyond max pages per sequence
    assert B.spec_pool_reserve(p, 1, 16 * 8) == 0
    assert B.spec_pool_reserve(p, 2, 17) == -2                 # pool exhausted: all or nothing
    assert B.spec_pool_block_table(p, 2) == []
    assert B.spec_pool_release(p, 1) == 0
    assert B.spec_pool_free_count(p) == 8
    assert B.spec_pool_commit(p, 0, 40, 0) == -4               # length beyond the held pages
    B.spec_pool_destroy(p)


def test_pool_prefix_sharing_refcounts(B):
    p = B.spec_pool_create(16, 16, 4, 8)
    B.spec_pool_reserve(p, 3, 64)                              # prefix holder: 4 pages
    assert B.spec_pool_share(p, 3, 4, 0) == 0
    assert B.spec_pool_share(p, 3, 4, 1) == 0
    assert B.spec_pool_refcount(p, 0) == 3
    B.spec_pool_reserve(p, 0, 80)                              # own page after the shared ones
    bt = B.spec_pool_block_table(p, 0)
    assert bt[:4] == [0, 1, 2, 3] and bt[4] not in (0, 1, 2, 3)
    B.spec_pool_release(p, 3)                                  # holder gone, users keep the pages
    assert B.spec_pool_refcount(p, 0) == 2
    B.spec_pool_release(p, 0)
    B.spec_pool_release(p, 1)
    assert B.spec_pool_free_count(p) == 16
    assert B.spec_pool_share(p, 0, 1, 0) == -1                 # src == dst
    B.spec_pool_destroy(p)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _agg_worker(rank, port, out):
    import torch.distributed as dist
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=2)
    ms, tok = bench.aggregate(10.0 + rank, 100 * (rank + 1))
    out.put((rank, ms, tok))
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_agg_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(60)
    assert res == [(0, 11.0, 300), (1, 11.0, 300)]


def test_rejection_sample_argument_contract(B):
    """spec_rejection_sample checks its arguments on the host before any CUDA
    call, with the error codes its declaration states (the pointers here are
    never dereferenced)."""
    fake = 1 << 20                                       # 16-byte aligned, never dereferenced
    ok = dict(logits_dev=fake, drafts_dev=fake, q_dev=None, u_accept_dev=fake, u_sample_dev=fake, n_seq=2, K=3,
              vocab=1024, temperature=1.0, out_accepted_dev=fake, out_token_dev=fake)
    cases = [
        (dict(logits_dev=None), -1), (dict(u_sample_dev=None), -1), (dict(out_token_dev=None), -1),
        (dict(drafts_dev=None), -1),                     # K > 0 needs drafts and acceptance uniforms
        (dict(n_seq=0), -1), (dict(K=-1), -1), (dict(vocab=2), -1),
        (dict(temperature=0.0), -1), (dict(temperature=float("nan")), -1),
        (dict(vocab=1022), -6), (dict(vocab=262_148), -6),
        (dict(logits_dev=fake + 4), -1),                 # logits must be 16-byte aligned
    ]
    for change, code in cases:
        with pytest.raises(B.SpecError) as e:
            B.spec_rejection_sample(**{**ok, **change})
        assert e.value.code == code, (change, str(e.value))
