"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from maxsim_scoring_gb300 import _native
from maxsim_scoring_gb300 import build as nvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return _native.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "maxsim.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(maxsim_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"maxsim_fwd", "maxsim_fwd_varlen", "maxsim_bwd", "maxsim_fwd_int8"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_native.SIGNATURES)


def test_status_strings_and_version(lib):
    for code in range(7):
        assert _native.status_string(code) not in ("", "unknown status")
    assert _native.status_string(99) == "unknown status"
    assert lib.maxsim_version() >= 100


FAKE = 0x10000  # 16-byte aligned fake device address: never dereferenced on the host


def fwd(lib, **kw):
    args = dict(Q=FAKE, D=FAKE, dtype=0, Nq=2, Lq=32, Nd=3, Ld=100, dim=128, q_mask=None, d_mask=None,
                scores=FAKE, argmax=None, ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return lib.maxsim_fwd(*args.values())


def test_fwd_host_validation(lib):
    assert fwd(lib, dtype=7) == 1
    assert fwd(lib, Nq=-1) == 1
    assert fwd(lib, dim=0) == 1
    assert fwd(lib, dim=24) == 2          # not a multiple of 16
    assert fwd(lib, dim=512) == 2         # beyond the supported width
    assert fwd(lib, scores=None) == 1
    assert fwd(lib, Q=FAKE + 8) == 1      # misaligned operand
    assert fwd(lib, Nq=0) == 0            # nothing to do: no launch, no device needed
    assert fwd(lib, Nd=0) == 0
    assert fwd(lib, Lq=40) == 5           # needs workspace (query rows are repacked), none given


def test_varlen_and_bwd_host_validation(lib):
    v = lib.maxsim_fwd_varlen
    assert v(FAKE, None, 32, FAKE, None, 100, 0, 2, 3, 128, None, None, FAKE, None, FAKE, 1 << 20, None) == 1
    assert v(FAKE, None, 32, FAKE, FAKE, -1, 0, 2, 3, 128, None, None, FAKE, None, FAKE, 1 << 20, None) == 1
    assert v(FAKE, None, 32, FAKE, FAKE, 100, 0, 2, 3, 128, None, None, FAKE, None, None, 0, None) == 5
    b = lib.maxsim_bwd
    assert b(FAKE, FAKE, 0, 2, 8, 3, 10, 128, None, None, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 20, None) == 1
    assert b(FAKE, FAKE, 0, 2, 8, 3, 10, 128, None, FAKE, FAKE, FAKE, FAKE, None, None, None, 0, None) == 5
    assert b(FAKE, FAKE, 3, 2, 8, 3, 10, 128, None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 20, None) == 1


def test_score_pairs_host_validation(lib):
    sp = lib.maxsim_score_pairs_packed
    # Q, cu_q, max_lq, D, cu_d, total_d, dtype, Nq, Nd, dim, q_mask, d_mask, pairs, n, scores, argmax, ws, bytes, stream
    assert sp(FAKE, None, 32, FAKE, FAKE, 100, 0, 2, 3, 128, None, None, FAKE, 0, FAKE, None, None, 0, None) == 0
    assert sp(FAKE, None, 32, FAKE, FAKE, 100, 0, 2, 3, 128, None, None, None, 5, FAKE, None, FAKE, 1 << 20, None) == 1
    assert sp(FAKE, None, 32, FAKE, None, 100, 0, 2, 3, 128, None, None, FAKE, 5, FAKE, None, FAKE, 1 << 20, None) == 1
    assert sp(FAKE, None, 32, FAKE, FAKE, 100, 2, 2, 3, 128, None, None, FAKE, 5, FAKE, None, FAKE, 1 << 20, None) == 1
    assert sp(FAKE, None, 32, FAKE, FAKE, 100, 0, 2, 3, 128, None, None, FAKE, 5, FAKE, None, None, 0, None) == 5
    assert sp(FAKE, None, 600, FAKE, FAKE, 100, 0, 2, 3, 128, None, None, FAKE, 5, FAKE, None, FAKE, 1 << 30,
              None) == 2                                            # one query per unit: at most 512 rows


def test_workspace_sizes(lib):
    ws = lib.maxsim_workspace_size
    assert ws(0, 32, 32, 100, 180, 128) == 0                      # aligned query length, no chunks
    assert ws(0, 2, 40, 3, 100, 128) >= 2 * 64 * 128 * 2          # padded to 64 rows per query
    assert ws(0, 1, 1024, 10, 1024, 128) >= 2 * 1 * 10 * 4        # two 512-row chunks of partial scores
    assert ws(1, 32, 32, 1000, 50000, 128) > 0                    # varlen always repacks the queries
    assert ws(2, 4, 8, 3, 10, 128) >= 4 * (3 + 4 + 31 + 96)      # counts, bases, row_ptr, col
    assert ws(4, 32, 32, 1000, 5000, 128) >= ws(1, 32, 32, 1000, 50000, 128) + 4 * (32 * 4 + 5000)  # + grouping
    assert ws(99, 1, 1, 1, 1, 16) == ctypes.c_size_t(-1).value
    assert ws(0, -1, 1, 1, 1, 16) == ctypes.c_size_t(-1).value


def test_chamfer_host_validation(lib):
    f, b = lib.maxsim_chamfer_fwd, lib.maxsim_chamfer_bwd
    # P, Q, B, N, M, dim, dist_p, idx_p, dist_q, idx_q, loss, ws, bytes, stream
    need = lib.maxsim_workspace_size(5, 2, 100, 70, 0, 3)
    assert f(FAKE, FAKE, 0, 100, 70, 3, None, None, None, None, None, None, 0, None) == 0   # nothing to do
    assert f(FAKE, FAKE, 2, 100, 70, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 1  # dim 0
    assert f(FAKE, FAKE, 2, 100, 70, 9, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 2  # dim > 8
    assert f(FAKE, FAKE, 2, -1, 70, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 1
    assert f(FAKE, FAKE, 2, 100, 70, 3, FAKE, FAKE, FAKE, FAKE, None, FAKE, need, None) == 1  # no loss
    assert f(FAKE, None, 2, 100, 70, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 1  # no Q
    assert f(FAKE + 2, FAKE, 2, 100, 70, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 1  # misaligned
    assert f(FAKE, FAKE, 2, 100, 70, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, None) == 5
    assert f(FAKE, FAKE, 2, 100, 70, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 16, need, None) == 5  # ws alignment
    # P, Q, B, N, M, dim, idx_p, idx_q, grad, dP, dQ, ws, bytes, stream
    nb = lib.maxsim_workspace_size(6, 2, 100, 70, 0, 3)
    assert b(FAKE, FAKE, 2, 0, 0, 3, None, None, None, None, None, None, 0, None) == 0
    assert b(FAKE, FAKE, 2, 100, 70, 3, FAKE, FAKE, None, FAKE, FAKE, FAKE, nb, None) == 1  # no grad
    assert b(FAKE, FAKE, 2, 100, 70, 3, FAKE, None, FAKE, FAKE, FAKE, FAKE, nb, None) == 1  # no idx_q
    assert b(FAKE, FAKE, 2, 100, 70, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, nb - 1, None) == 5


def test_chamfer_workspace_sizes(lib):
    ws = lib.maxsim_workspace_size
    B, N, M = 2, 5000, 9000
    # per direction: one (min, sub-tile) pair per source and 4096-target span
    spans_p, spans_q = -(-M // 4096), -(-N // 4096)
    assert ws(5, B, N, M, 0, 8) >= 8 * B * (N * spans_p + M * spans_q)
    # dim <= 4 (tensor cores): two 64-byte operand rows per point, padded
    assert ws(5, B, N, M, 0, 3) >= 2 * 64 * B * (N + M)
    assert ws(5, B, N, M, 0, 4) == ws(5, B, N, M, 0, 1)
    # two key / value buffers, the row pointers
    assert ws(6, B, N, M, 0, 3) >= 16 * B * (N + M) + 4 * (B * (N + M) + 1)
    assert ws(6, 0, 0, 0, 0, 3) == 0
    assert ws(5, 1, 1, 1, 0, 0) == ctypes.c_size_t(-1).value


def test_topk_and_two_stage_host_validation(lib):
    t = lib.maxsim_topk
    # scores, rows, n, k, idx, vals, stream
    assert t(FAKE, 0, 10, 3, None, None, None) == 0       # nothing to do
    assert t(FAKE, 2, 10, 11, FAKE, None, None) == 1      # k > n
    assert t(FAKE, 2, 10000, 5000, FAKE, None, None) == 2  # k above 4096
    assert t(None, 2, 10, 3, FAKE, None, None) == 1
    assert t(FAKE + 2, 2, 10, 3, FAKE, None, None) == 1   # misaligned
    ts = lib.maxsim_two_stage_topk
    need = lib.maxsim_workspace_size(7, 4, 32, 1000, 64, 128)
    assert need != ctypes.c_size_t(-1).value and need >= 4 * 1000 * 4
    # Q8, qs, D8, ds, Q16, D16, dtype, Nq, Lq, Nd, Ld, dim, k1, k, idx, scores, s8, cand, ws, bytes, stream
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 32, 1000, 64, 128, 100, 10, FAKE, None, None, None, FAKE, need,
            None]
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return ts(*a)
    assert call(a13=0) == 0              # k = 0: nothing to do
    assert call(a12=1001) == 1           # k1 > Nd
    assert call(a13=101) == 1            # k > k1
    assert call(a11=48) == 2             # dim not a multiple of 32
    assert call(a8=600) == 2             # the rescoring stage takes up to 512 query rows
    assert call(a6=5) == 1               # dtype
    assert call(a14=None) == 1           # no output
    assert call(a19=1024) == 5            # far too small
    assert call(a18=FAKE + 16) == 5      # workspace alignment


def test_streamed_host_validation(lib):
    f = lib.maxsim_fwd_streamed
    need = lib.maxsim_workspace_size(8, 1, 32, 20000, 1024, 128)
    assert need >= 2 * 20000 * 1024 * 128 * 2          # two device blocks
    assert lib.maxsim_workspace_size(8, 1, 32, 20000, 1024, 128) == need  # independent of the corpus size
    # Q, D_host, dtype, Nq, Lq, Nd, Ld, dim, block, q_mask, scores, ws, bytes, stream
    assert f(FAKE, FAKE, 0, 1, 32, 0, 1024, 128, 20000, None, FAKE, None, 0, None) == 0  # no documents
    assert f(FAKE, FAKE, 0, 1, 32, 5, 1024, 128, 0, None, FAKE, FAKE, need, None) == 1   # block of 0
    assert f(FAKE, FAKE, 0, 1, 32, 5, 1024, 128, 20000, None, None, FAKE, need, None) == 1
    assert f(FAKE, None, 0, 1, 32, 5, 1024, 128, 20000, None, FAKE, FAKE, need, None) == 1
    assert f(FAKE, FAKE, 0, 1, 32, 5, 1024, 24, 20000, None, FAKE, FAKE, need, None) == 2  # dim
    assert f(FAKE, FAKE, 0, 1, 32, 50000, 1024, 128, 20000, None, FAKE, FAKE, 1024, None) == 5


def test_bwd_varlen_host_validation(lib):
    b = lib.maxsim_bwd_varlen
    need = lib.maxsim_workspace_size(9, 4, 32, 10, 1000, 128)
    assert need >= 4 * (1000 + 1) + 4 * 4 * 10 * 32
    # Q, cu_q, max_lq, D, cu_d, total_d, max_ld, dtype, Nq, Nd, dim, q_mask, argmax, g, dQ, dD, rp, col, ws, bytes, st
    args = [FAKE, None, 32, FAKE, FAKE, 1000, 300, 0, 4, 10, 128, None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, need,
            None]
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return b(*a)
    assert call(a4=None) == 1            # no document offsets
    assert call(a12=None) == 1           # no argmax
    assert call(a7=3) == 1               # dtype
    assert call(a10=24) == 2             # dim
    assert call(a6=60000) == 2           # a document histogram beyond shared memory
    assert call(a19=64) == 5             # workspace
    assert call(a15=FAKE + 4) == 1       # misaligned gradient


def test_varlen_streamed_host_validation(lib):
    f = lib.maxsim_fwd_varlen_streamed
    cu = (ctypes.c_int32 * 4)(0, 100, 100, 350)            # host offsets: 3 documents, 350 rows
    bad = (ctypes.c_int32 * 4)(0, 100, 90, 350)            # decreasing
    need = lib.maxsim_workspace_size(10, 2, 32, 3, 1000, 128)
    # Q, cu_q, max_lq, D_host, cu_host, total_d, dtype, Nq, Nd, dim, q_mask, block_docs, block_tokens, scores, ws, n, st
    p_cu = ctypes.cast(cu, ctypes.c_void_p).value
    p_bad = ctypes.cast(bad, ctypes.c_void_p).value
    assert f(FAKE, None, 32, FAKE, p_cu, 350, 0, 2, 3, 128, None, 3, 1000, FAKE, FAKE, need, None) != 1
    assert f(FAKE, None, 32, FAKE, p_bad, 350, 0, 2, 3, 128, None, 3, 1000, FAKE, FAKE, need, None) == 1
    assert f(FAKE, None, 32, FAKE, p_cu, 349, 0, 2, 3, 128, None, 3, 1000, FAKE, FAKE, need, None) == 1
    assert f(FAKE, None, 32, FAKE, p_cu, 350, 0, 2, 3, 128, None, 3, 200, FAKE, FAKE, need, None) == 2  # 250 > 200
    assert f(FAKE, None, 32, FAKE, p_cu, 350, 0, 2, 3, 128, None, 0, 1000, FAKE, FAKE, need, None) == 1
    assert f(FAKE, None, 32, FAKE, p_cu, 350, 0, 2, 3, 128, None, 3, 1000, FAKE, FAKE, 64, None) == 5
    assert f(FAKE, None, 32, FAKE, None, 350, 0, 2, 3, 128, None, 3, 1000, FAKE, FAKE, need, None) == 1
