"""The hot path replayed from a CUDA graph.

A serving loop launches the same three calls every step; capturing them once in
a CUDA graph removes the host cost of each launch (argument checks, tensor-map
encoding, the occupancy query).  Every call is stream-ordered and allocates
nothing, so the projection, the norm/RoPE pass and the KV-cache call can be
captured on torch's capture stream and replayed.  The one-time lookups the calls
make (the device's SM count, the KV status word) happen in an eager call first,
as the header asks.  The replayed results must match the oracle, and replaying
again must give the same bytes.
"""
import numpy as np
import pytest
import torch

from parity_util import as_f64, check_kv, check_qkv, qkv_reference
from rope_attention_gb300 import native, runner, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", [native.RA_LAYOUT_BSD, native.RA_LAYOUT_NBSD], ids=["bsd", "nbsd"])
def test_step_replays_from_a_cuda_graph(layout):
    # across-heads norm + RoPE in BSD or NBSd (the pipelined second passes; NBSd's takes a
    # tensor map as a kernel parameter), V2 int8 PA_BNSD (pipelined KV kernel)
    qcase = synth.make_qkv("graph_q", 41, S=300, H=256, num_heads=4, num_kv_heads=4, head_dim=64)
    kcase = synth.make_kv("graph_kv", 42, variant=2, B=2, N=8, S=40, Dkv=192, Dv=128, block_size=32,
                          block_num=4, quant_k=True, quant_v=True, skip_frac=0.1)
    q, k = runner.QkvRun(qcase, layout=layout), runner.KvRun(kcase)
    as_bsd = (lambda t: t) if layout == native.RA_LAYOUT_BSD else \
        (lambda t: t.permute(1, 0, 2).reshape(qcase.T, qcase.I))
    q.project()
    q.norm_rope()
    k.run()
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        q.project()
        q.norm_rope()
        k.run()

    # start from clean outputs, so that what is checked is what the replay wrote
    q.out.zero_()
    k.k_cache.copy_(runner.to_dev(kcase.k_cache))
    k.ckv_cache.copy_(runner.to_dev(kcase.ckv_cache))
    graph.replay()
    torch.cuda.synchronize()
    assert q.status() == 0 and native.kv_rms_norm_rope_cache_status() == 0
    check_qkv(qcase, as_f64(as_bsd(q.out)), qkv_reference(qcase), "graph replay")
    check_kv(kcase, k, "graph replay")

    first = (q.out.clone(), k.k_cache.clone(), k.ckv_cache.clone())
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(first, (q.out, k.k_cache, k.ckv_cache)):
        assert torch.equal(a, b)
    assert not np.any(np.isnan(as_f64(q.out)))
