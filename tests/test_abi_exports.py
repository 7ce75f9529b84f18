"""The C-ABI library builds, loads without a GPU and exports every function
include/phs.h declares; the Python binding declares exactly those."""
import ctypes
import os
import re

import pytest

import paged_hybrid_sliding_gb300 as phs
from paged_hybrid_sliding_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "phs.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(phs_[a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def so():
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_expected_calls():
    names = declared_functions()
    for n in ["phs_kv_append_paged", "phs_kv_append_ring", "phs_kv_quant_int8_block32",
              "phs_attn_decode_full_paged", "phs_attn_decode_swa_ring",
              "phs_attn_decode_hybrid_stack"]:
        assert n in names


def test_library_exports_every_declared_symbol(so):
    for name in declared_functions():
        assert hasattr(so, name), f"{name} not exported"


def test_binding_covers_header(so):
    assert sorted(_lib.EXPORTED) == declared_functions()


def test_host_only_calls(so):
    lib = phs.lib()
    assert lib.phs_version() >= 1
    assert lib.phs_status_str(0) == b"ok"
    assert b"shared" in lib.phs_status_str(-4)
    f, w = phs.hybrid_kv_tokens([1, 0, 0], [10, 200, 128], 128)
    assert f == 338 and w == 2 * (10 + 128 + 128)


def test_hybrid_kv_tokens_matches_oracle():
    import numpy as np

    import oracle
    import synth
    wl = synth.hybrid_stack()
    lf = wl.extra["layer_is_full"]
    f, s = phs.hybrid_kv_tokens(lf, wl.n_after, 128)
    assert f + s == oracle.kv_tokens_stored(lf, wl.n_after, 128)
    assert f == oracle.kv_tokens_stored(lf * 0 + lf, wl.n_after, 128) - s
    allf = oracle.kv_tokens_stored(np.ones(70, np.int32), wl.n_after, 128)
    assert abs((f + s) / allf - 1 / 7) / (1 / 7) < 0.05


def test_int8_pool_codes_reads_the_stored_form():
    """Int8Pool.codes() undoes the stored form include/phs.h states for
    phs_int8_pool: byte x + 128; K token-major; V per 16-token half hf, one
    16-byte row per head dim, byte p holding token 16 hf + 2(p/4) + (p%2) +
    8((p/2)%2).  The stored pool is written here element by element from
    that statement."""
    import torch
    g = torch.Generator().manual_seed(7)
    n, h, D = 2, 3, 8
    kc = torch.randint(-127, 128, (n, h, 32, D), generator=g)
    vc = torch.randint(-127, 128, (n, h, 32, D), generator=g)
    k = torch.empty((n, h, 32, D), dtype=torch.uint8)
    v = torch.empty((n, h, 2, D, 16), dtype=torch.uint8)
    for i in range(n):
        for j in range(h):
            for t in range(32):
                for d in range(D):
                    k[i, j, t, d] = int(kc[i, j, t, d]) + 128
            for d in range(D):
                for hf in range(2):
                    for p in range(16):
                        t = 16 * hf + 2 * (p // 4) + p % 2 + 8 * ((p // 2) % 2)
                        v[i, j, hf, d, p] = int(vc[i, j, t, d]) + 128
    pool = phs.Int8Pool(k, v, torch.zeros(n, h), torch.zeros(n, h))
    gk, gv = pool.codes()
    assert gk.dtype == torch.int8 and torch.equal(gk.long(), kc)
    assert gv.dtype == torch.int8 and torch.equal(gv.long(), vc)
    gk1, gv1 = pool.codes(torch.tensor([1]))
    assert torch.equal(gk1.long(), kc[1:]) and torch.equal(gv1.long(), vc[1:])
    assert sorted(phs.VT_TOKEN) == list(range(16))
