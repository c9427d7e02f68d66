"""maxsim_fwd_streamed (out-of-core corpus in host memory) against the
device-resident forward, bit for bit, and against the oracle."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from maxsim_scoring_gb300 import ops
from tests.gpu_util import TORCH_DT, assert_scores, dev_bits

pytestmark = pytest.mark.gpu


def host_bits(bits, dtype, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DT[dtype])
    return t.pin_memory() if pin else t


@pytest.mark.parametrize("Nq,Lq,Nd,Ld,block,dtype", [(3, 32, 1000, 200, 128, "bf16"), (1, 40, 777, 64, 100, "f16"),
                                                     (2, 600, 90, 300, 16, "bf16"), (1, 32, 50, 1024, 1000, "f16")])
def test_streamed_equals_the_device_forward(Nq, Lq, Nd, Ld, block, dtype):
    Q = datagen.gaussian_rows(61, 1, Nq * Lq, 128, dtype).reshape(Nq, Lq, 128)
    D = datagen.gaussian_rows(61, 2, Nd * Ld, 128, dtype).reshape(Nd, Ld, 128)
    Qd = dev_bits(Q, dtype)
    Dh = host_bits(D, dtype)  # alive until the stream has passed the call
    got = ops.maxsim_fwd_streamed(Qd, Dh, block_docs=block)
    want, _ = ops.maxsim_fwd(Qd, dev_bits(D, dtype))
    assert ops.device_status() == 0
    assert torch.equal(got, want)
    docs = np.arange(0, Nd, max(1, Nd // 40))
    ref, _, _ = oracle.fwd_dense(Q, D, dtype, docs=docs)
    assert_scores(got[:, torch.from_numpy(docs)], ref, Lq)


def test_streamed_pageable_memory_and_query_mask():
    Nq, Lq, Nd, Ld = 2, 32, 300, 100
    Q = datagen.gaussian_rows(67, 1, Nq * Lq, 128, "f16").reshape(Nq, Lq, 128)
    D = datagen.gaussian_rows(67, 2, Nd * Ld, 128, "f16").reshape(Nd, Ld, 128)
    qm = (np.random.default_rng(67).random((Nq, Lq)) > 0.3).astype(np.uint8)
    Qd = dev_bits(Q, "f16")
    Dh = host_bits(D, "f16", pin=False)
    got = ops.maxsim_fwd_streamed(Qd, Dh, torch.from_numpy(qm).cuda(), block_docs=64)
    want, _ = ops.maxsim_fwd(Qd, dev_bits(D, "f16"), torch.from_numpy(qm).cuda())
    assert ops.device_status() == 0
    assert torch.equal(got, want)


def test_streamed_calls_back_to_back_reuse_the_buffers():
    # two calls enqueued without a host sync in between, on the same stream
    Q = datagen.gaussian_rows(71, 1, 32, 128, "bf16").reshape(1, 32, 128)
    D1 = datagen.gaussian_rows(71, 2, 500 * 64, 128, "bf16").reshape(500, 64, 128)
    D2 = datagen.gaussian_rows(71, 3, 500 * 64, 128, "bf16").reshape(500, 64, 128)
    Qd = dev_bits(Q, "bf16")
    D1h, D2h = host_bits(D1, "bf16"), host_bits(D2, "bf16")
    a = ops.maxsim_fwd_streamed(Qd, D1h, block_docs=100)
    b = ops.maxsim_fwd_streamed(Qd, D2h, block_docs=100)
    wa, _ = ops.maxsim_fwd(Qd, dev_bits(D1, "bf16"))
    wb, _ = ops.maxsim_fwd(Qd, dev_bits(D2, "bf16"))
    assert ops.device_status() == 0
    assert torch.equal(a, wa) and torch.equal(b, wb)


@pytest.mark.parametrize("Nq,block_docs,block_tokens", [(4, 50, 4000), (1, 1000, 300), (3, 7, 100000), (2, 10000, 1 << 22)])
def test_varlen_streamed_equals_the_device_forward(Nq, block_docs, block_tokens):
    rng = np.random.default_rng(107 + Nq)
    dtype, dim, Lq = "f16", 128, 32
    lens = rng.integers(0, 301, size=600)
    lens[::37] = 0
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    D = datagen.gaussian_rows(107, 2, int(cu[-1]), dim, dtype)
    Q = datagen.gaussian_rows(107, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    Qd = dev_bits(Q, dtype)
    Dh = host_bits(D, dtype)
    cu_h = torch.from_numpy(cu)
    got = ops.maxsim_fwd_varlen_streamed(Qd, None, Lq, Dh, cu_h, block_docs=block_docs, block_tokens=block_tokens)
    want, _ = ops.maxsim_fwd_varlen(Qd, None, Lq, dev_bits(D, dtype), torch.from_numpy(cu).cuda())
    assert ops.device_status() == 0
    assert torch.equal(got, want)


def test_varlen_streamed_packed_queries_and_document_too_long():
    rng = np.random.default_rng(109)
    dtype, dim = "bf16", 64
    qlens = np.array([5, 32, 17])
    cu_q = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    lens = rng.integers(1, 200, size=90)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Q = datagen.gaussian_rows(109, 1, int(cu_q[-1]), dim, dtype)
    D = datagen.gaussian_rows(109, 2, int(cu[-1]), dim, dtype)
    Qd, cq = dev_bits(Q, dtype), torch.from_numpy(cu_q).cuda()
    Dh, cu_h = host_bits(D, dtype), torch.from_numpy(cu)
    got = ops.maxsim_fwd_varlen_streamed(Qd, cq, 32, Dh, cu_h, block_docs=16, block_tokens=1000)
    want, _ = ops.maxsim_fwd_varlen(Qd, cq, 32, dev_bits(D, dtype), torch.from_numpy(cu).cuda())
    assert ops.device_status() == 0
    assert torch.equal(got, want)
    with pytest.raises(Exception):  # a document longer than a block
        ops.maxsim_fwd_varlen_streamed(Qd, cq, 32, Dh, cu_h, block_docs=16, block_tokens=int(lens.max()) - 1)
