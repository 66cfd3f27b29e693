"""gqa_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (a host program whose memory is all in its own pool, a
decode loop that must not let cudaMalloc synchronise the device).  Called
through the C ABI on three calls in a row, of different shapes (the last one
small enough for the direct kernel); each output must
match the fp64 oracle, and gqa_decode_attention's output, within the parity
tolerance.  Collected last on purpose, so that a run stopping at the first
failure has run every other test already."""
import ctypes

import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from gqa_decode_attention_02_gb300 import _lib
from helpers import TOL, assert_close, small, to, ulp

pytestmark = pytest.mark.gpu


def _entry():
    f = _lib.lib().gqa_decode_attention_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(_lib.Shape)] + [ctypes.c_void_p] * 8
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_oracle_and_workspace_entry_point_on_calls_in_a_row(gpu):
    f = _entry()
    cases = [
        # ragged bf16 batch with long contexts: split sequences, merged pieces
        small(B=6, T=1, N=32, K=8, H=128, dtype="bf16", ctx=(5, 700, 4097, 33, 16, 2000),
              seed=61),
        # then an fp16 H=64 batch of another shape, on the same static scratch
        small(B=5, T=1, N=14, K=2, H=64, dtype="f16", ctx=(1, 295, 1024, 17, 3000), seed=62),
        # and a small call, served by the direct kernel (no scratch used)
        small(B=2, T=1, N=14, K=2, H=64, dtype="f16", ctx=(295, 40), seed=63),
    ]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for w in cases:
        wd = to(w, gpu)
        ref = gq.decode_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                                  wd.context_lens)
        out = torch.full_like(wd.q[0], float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device=gpu)
        shape = _lib.make_shape(wd.q[0], wd.k_cache[0], wd.block_tables, None)
        rc = f(ctypes.byref(shape), _p(wd.q[0]), _p(wd.k_cache[0]), _p(wd.v_cache[0]),
               _p(wd.block_tables), _p(wd.context_lens), _p(out), _p(st), stream)
        assert rc == 0, _lib.status_string(rc)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        want, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                   w.context_lens, w.dtype)
        assert_close(out.double().cpu().numpy(), want, w.dtype, "noalloc vs oracle")
        a = out.double().cpu().numpy()
        b = ref.double().cpu().numpy()
        assert np.isfinite(a).all()
        lim = np.maximum(TOL[w.dtype], ulp(b, w.dtype))
        assert (np.abs(a - b) <= lim).all(), float(np.abs(a - b).max())


def test_noalloc_rejects_bad_shapes_before_touching_the_gpu(gpu):
    f = _entry()
    shape = _lib.Shape(B=2, T=2, N=8, K=2, H=64, block_size=16, num_blocks=4,
                       max_blocks_per_seq=2, dtype=0, scale=0.0, flags=0)
    fake = ctypes.c_void_p(16)
    assert f(ctypes.byref(shape), fake, fake, fake, fake, fake, fake, None, None) == 2  # T != 1
    assert f(None, fake, fake, fake, fake, fake, fake, None, None) == 1
    # 64 query rows per KV head pick the tensor-memory kernel, whose scratch
    # (256 KiB + 132 KiB per SM) exceeds the fixed 8 MiB on GPUs of more than
    # 60 SMs: rejected before any launch
    mqa = _lib.Shape(B=2, T=1, N=64, K=1, H=128, block_size=16, num_blocks=4,
                     max_blocks_per_seq=2, dtype=1, scale=0.0, flags=0)
    sms = torch.cuda.get_device_properties(gpu).multi_processor_count
    want = 5 if (256 << 10) + sms * (132 << 10) > (8 << 20) else 0
    if want:
        assert f(ctypes.byref(mqa), fake, fake, fake, fake, fake, fake, None, None) == want
