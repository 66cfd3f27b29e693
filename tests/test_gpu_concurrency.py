"""Attention calls that overlap on the GPU.

Split segments are merged by whichever piece finishes last (an atomic ticket),
so no thread block waits for another and nothing depends on which thread
blocks are resident at the same time.  These tests run calls on two streams at
once -- each with its own workspace, the binding's per-stream default or the
caller's -- and next to a long GEMM that holds SMs, and check every output
against the fp64 oracle, the device status, and bit-identity with the same
call run alone."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from helpers import assert_close, small, to

pytestmark = pytest.mark.gpu


def _oracle(w):
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, w.dtype)
    assert (err == 0).all()
    return out


def _cases():
    # long ragged contexts (split segments on many CTAs): the warp-level
    # kernel (4 rows per KV head) and the tensor-memory kernel (40 rows)
    a = small(B=5, T=1, N=32, K=8, H=128, dtype="bf16", ctx=(30000, 5, 17000, 4097, 1),
              seed=91)
    b = small(B=4, T=5, N=64, K=8, H=128, dtype="bf16", ctx=(20000, 600, 9000, 5), seed=92)
    return a, b


def _call(wd, stream, workspace=None, status=None):
    fn = gq.decode_attention if wd.T == 1 else gq.verify_attention
    with torch.cuda.stream(stream):
        return fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens,
                  workspace=workspace, status=status, stream=stream)


@pytest.mark.parametrize("explicit_workspace", [False, True])
def test_two_streams_at_once(gpu, explicit_workspace):
    wa, wb = _cases()
    da, db = to(wa, gpu), to(wb, gpu)
    sa, sb = torch.cuda.Stream(gpu), torch.cuda.Stream(gpu)
    st = torch.zeros(2, dtype=torch.int32, device=gpu)
    ws = [None, None]
    if explicit_workspace:
        ws = [torch.zeros(gq.attention_workspace_size(d.q[0], d.k_cache[0], d.block_tables),
                          dtype=torch.uint8, device=gpu) for d in (da, db)]
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):  # calls alternate between the streams without syncing
        outs.append((_call(da, sa, ws[0], st[0:1]), _call(db, sb, ws[1], st[1:2])))
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    ra, rb = _oracle(wa), _oracle(wb)
    for oa, ob in outs:
        assert_close(oa.double().cpu().numpy(), ra, "bf16", "stream A")
        assert_close(ob.double().cpu().numpy(), rb, "bf16", "stream B")
        assert torch.equal(oa, outs[0][0]) and torch.equal(ob, outs[0][1])
    # the same calls alone on the default stream give the same bits
    alone = _call(da, torch.cuda.current_stream(gpu))
    torch.cuda.synchronize()
    assert torch.equal(alone, outs[0][0])


def test_attention_next_to_a_gemm_that_holds_sms(gpu):
    """A long GEMM on another stream occupies SMs while the attention grid
    launches, so not all of its thread blocks can be resident at once."""
    wa, wb = _cases()
    da, db = to(wa, gpu), to(wb, gpu)
    ref_a = _call(da, torch.cuda.current_stream(gpu))
    ref_b = _call(db, torch.cuda.current_stream(gpu))
    torch.cuda.synchronize()
    busy, side = torch.cuda.Stream(gpu), torch.cuda.Stream(gpu)
    x = torch.randn(8192, 8192, dtype=torch.bfloat16, device=gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    torch.cuda.synchronize()
    with torch.cuda.stream(busy):
        for _ in range(4):
            y = x @ x  # noqa: F841  (keeps SMs busy)
    got_a = _call(da, side, status=st)
    got_b = _call(db, side, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(got_a, ref_a) and torch.equal(got_b, ref_b)
    assert_close(got_b.double().cpu().numpy(), _oracle(wb), "bf16", "next to a GEMM")


def test_direct_kernel_next_to_a_split_one_on_two_streams(gpu):
    """A small call (the direct kernel: one CTA per sequence and KV head) and
    a large one (the persistent kernel, split segments) overlapping on two
    streams, three times without syncing: every output equals the oracle's and
    the same call run alone."""
    small_w = small(B=3, T=1, N=14, K=2, H=64, dtype="f16", ctx=(1, 295, 1000), seed=93)
    big_w, _ = _cases()
    ds, db = to(small_w, gpu), to(big_w, gpu)
    assert gq.attention_engine(small_w.q[0], small_w.k_cache[0], small_w.block_tables) == "direct"
    sa, sb = torch.cuda.Stream(gpu), torch.cuda.Stream(gpu)
    st = torch.zeros(2, dtype=torch.int32, device=gpu)
    torch.cuda.synchronize()
    outs = [(_call(ds, sa, status=st[0:1]), _call(db, sb, status=st[1:2])) for _ in range(3)]
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    rs, rb = _oracle(small_w), _oracle(big_w)
    for os_, ob in outs:
        assert_close(os_.double().cpu().numpy(), rs, "f16", "direct, stream A")
        assert_close(ob.double().cpu().numpy(), rb, "bf16", "persistent, stream B")
        assert torch.equal(os_, outs[0][0]) and torch.equal(ob, outs[0][1])
    alone = _call(ds, torch.cuda.current_stream(gpu))
    torch.cuda.synchronize()
    assert torch.equal(alone, outs[0][0])


def test_binding_keeps_one_workspace_per_stream(gpu):
    from gqa_decode_attention_02_gb300 import _lib

    wa, _ = _cases()
    da = to(wa, gpu)
    sa, sb = torch.cuda.Stream(gpu), torch.cuda.Stream(gpu)
    _call(da, sa)
    _call(da, sb)
    torch.cuda.synchronize()
    keys = {k for k in _lib._ws_cache if k[2] == "attention"}
    assert (gpu.index or 0, int(sa.cuda_stream), "attention") in keys
    assert (gpu.index or 0, int(sb.cuda_stream), "attention") in keys
    wsa = _lib._ws_cache[(gpu.index or 0, int(sa.cuda_stream), "attention")]
    wsb = _lib._ws_cache[(gpu.index or 0, int(sb.cuda_stream), "attention")]
    assert wsa.data_ptr() != wsb.data_ptr()
    # every call leaves its workspace's ticket region zero-filled
    for ws in (wsa, wsb):
        assert int(ws[: 256 * 1024].view(torch.int32).abs().sum().item()) == 0
    gq.reset_workspaces()
    assert not _lib._ws_cache
