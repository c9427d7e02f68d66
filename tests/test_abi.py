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
    assert ws(9, 1, 1, 1, 1, 16) == ctypes.c_size_t(-1).value
    assert ws(0, -1, 1, 1, 1, 16) == ctypes.c_size_t(-1).value
