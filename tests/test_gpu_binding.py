"""The binding's default workspaces: a call that passes none uses one kept per (device, stream, kind),
made zero-filled once and grown when a batch needs more, so repeated calls allocate nothing; under
CUDA-graph capture the binding refuses to make one."""
import numpy as np
import pytest

import workloads as W
from tests.gpu_util import DeviceBatch, host_bits

pytestmark = pytest.mark.gpu


def _cached(nv, kind):
    return [t for (dev, stream, k), t in nv._ws_cache.items() if k == kind]


def test_default_decode_workspace_is_reused_then_grown():
    import torch
    import paged_kv_attention_store_gb300 as nv
    nv.release_default_workspaces()
    small = W.make_decode("ws-small", 71, [700, 1500, 33], 32, 8, 128, 64)
    db = DeviceBatch(small)
    db.store()
    maxc = int(small.seq_lens.max())
    ws = torch.zeros(nv.nv_paged_decode_workspace_size(small.num_seqs, 32, 128, maxc), dtype=torch.uint8,
                     device="cuda")
    want = host_bits(nv.nv_paged_decode_attn(db.q, db.k_cache, db.v_cache, db.block_tables, db.seq_lens, small.scale,
                                             max_context_len=maxc, workspace=ws))
    outs = [host_bits(db.decode()) for _ in range(3)]
    for o in outs:
        assert np.array_equal(o, want)
    first = _cached(nv, "decode")
    assert len(first) == 1
    ptr = first[0].data_ptr()
    db.decode()
    assert [t.data_ptr() for t in _cached(nv, "decode")] == [ptr]        # reused, not reallocated
    # a batch needing more workspace grows it once, and still decodes correctly
    big = W.qwen8_decode(num_seqs=8)
    dbb = DeviceBatch(big)
    dbb.store()
    bmax = int(big.seq_lens.max())
    ws_b = torch.zeros(nv.nv_paged_decode_workspace_size(big.num_seqs, 32, 128, bmax), dtype=torch.uint8,
                       device="cuda")
    want_b = host_bits(nv.nv_paged_decode_attn(dbb.q, dbb.k_cache, dbb.v_cache, dbb.block_tables, dbb.seq_lens,
                                               big.scale, max_context_len=bmax, workspace=ws_b))
    assert np.array_equal(host_bits(dbb.decode()), want_b)
    grown = _cached(nv, "decode")
    assert len(grown) == 1 and grown[0].numel() >= ws_b.numel()
    assert np.array_equal(host_bits(db.decode()), want)                 # the small batch again, same result
    assert db.err() == 0 and dbb.err() == 0
    nv.release_default_workspaces()
    assert not nv._ws_cache


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_default_workspace_is_not_made_during_graph_capture():
    import torch
    import paged_kv_attention_store_gb300 as nv
    nv.release_default_workspaces()
    b = W.make_decode("ws-capture", 72, [900, 40], 32, 8, 128, 64)
    db = DeviceBatch(b)
    db.store()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with pytest.raises(ValueError, match="pass a workspace when capturing"):
            with torch.cuda.graph(g, stream=s):
                nv.nv_paged_decode_attn(db.q, db.k_cache, db.v_cache, db.block_tables, db.seq_lens, b.scale,
                                        max_context_len=int(b.seq_lens.max()))
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert not _cached(nv, "decode")
