"""Every mbarrier wait of the decode kernels is bounded: a wait that runs out
records PHS_ETIMEOUT in the status word, drains the warp's other copies in
flight and returns, so the context stays usable.  To make a wait run out
without a fault, the test builds a variant of the library from a patched
copy of the sources (never the product build): the wait limit is cut to
2 ms and the TMA producer of one warp skips both the copy and the arrival of
one stage, so that nothing is in flight for it and its consumer's wait
cannot complete.  Covered: the split-KV kernel and both SWA ring kernels,
the persistent one and the one-CTA-per-unit latency shape (the tensor-core
shared-prefix kernel is left out).  Other requests must come
out exactly as the product library computes them."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import paged_hybrid_sliding_gb300 as phs
import synth
from paged_hybrid_sliding_gb300 import _lib
from paged_hybrid_sliding_gb300 import build as phs_build
from gpu_util import dev

pytestmark = pytest.mark.gpu

PATCHES = {
    "phs_common.cuh": [("constexpr uint64_t kWaitLimitNs = 1000000000ull;",
                        "constexpr uint64_t kWaitLimitNs = 2000000ull;")],
    # split kernel: CTA (0, 0, 0), warp 0 never issues its chunk 1
    "phs_decode.cu": [("  auto issue = [&](int j) {  // lane 0 only\n",
                       "  auto issue = [&](int j) {  // lane 0 only\n"
                       "    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && "
                       "warp == 0 && j == 1) return;\n")],
    # SWA kernels: block 0, warp 0 never issues the second chunk of its
    # first unit (persistent kernel) or its second chunk (one CTA per unit)
    "phs_swa.cu": [("    if (!iu.ok) {\n",
                    "    if (blockIdx.x == 0 && warp == 0 && ik == 0 && ic == 1) {\n"
                    "    } else if (!iu.ok) {\n")],
    "phs_swa_chunk.cuh": [("  auto issue = [&](int jj) {  // lane 0: chunk warp + NW jj into stage jj % S\n",
                           "  auto issue = [&](int jj) {  // lane 0: chunk warp + NW jj into stage jj % S\n"
                           "    if (blockIdx.x == 0 && warp == 0 && jj == 1) return;\n")],
}


@pytest.fixture(scope="module")
def wait_lib(tmp_path_factory):
    phs_build.build()  # the product objects the variant links against
    d = tmp_path_factory.mktemp("wait_variant")
    src = os.path.join(phs_build.HERE, "csrc")
    for name in os.listdir(src):
        shutil.copy(os.path.join(src, name), d / name)
    for name, changes in PATCHES.items():
        text = (d / name).read_text()
        for old, new in changes:
            assert text.count(old) == 1, (name, old)
            text = text.replace(old, new)
        (d / name).write_text(text)
    nvcc = phs_build.nvcc_path()
    flags = [f if f != phs_build.CSRC else str(d) for f in phs_build._flags()]
    objs = []
    procs = []
    for name in ("phs_decode.cu", "phs_swa.cu"):
        o = str(d / (name[:-3] + ".o"))
        procs.append(subprocess.Popen([nvcc, *flags, "-c", str(d / name), "-o", o],
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT))
        objs.append(o)
    for p in procs:
        out, _ = p.communicate()
        assert p.returncode == 0, out.decode()[-3000:]
    keep = [os.path.join(phs_build.BUILD, n) for n in sorted(os.listdir(phs_build.BUILD))
            if n.endswith(".o") and n not in ("phs_decode.o", "phs_swa.o")]
    so = str(d / "libphs_wait_variant.so")
    subprocess.check_call([nvcc, *phs_build.ARCH, "-shared", "-Xlinker", "-Bsymbolic", "-o",
                           so, *objs, *keep])
    lib = ctypes.CDLL(so)
    for name in ("phs_attn_decode_full_paged", "phs_attn_decode_swa_ring"):
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = _lib._SIGS[name]
    return lib


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def test_split_kernel_wait_runs_out_and_returns(wait_lib):
    B, Hq, Hkv, D = 3, 32, 8, 128
    lens = np.array([2000, 777, 3001], np.int32)
    bt, npg = synth.block_tables_from_permutation(synth.pages_needed(lens), 5)
    pool = phs.PagedPool(synth.normal_bf16((npg, Hkv, 16, D), 6, device="cuda"),
                         synth.normal_bf16((npg, Hkv, 16, D), 7, device="cuda"))
    q = synth.normal_bf16((B, Hq, D), 8, device="cuda")
    ms = int(lens.max())
    ref = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), ms, out_dtype=torch.float32)
    out = torch.zeros_like(ref)
    ws = torch.empty(phs.decode_workspace_bytes(B, Hq, Hkv, D, ms), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pc = pool.c()
    btd, sld = dev(bt), dev(lens)
    rc = wait_lib.phs_attn_decode_full_paged(
        _vp(q), Hq, ctypes.byref(pc), _vp(btd), bt.shape[1], _vp(sld), ms, None, None, 0, None,
        B, 1 / np.sqrt(D), 0, _vp(out), 1, _vp(ws), ws.numel(), None, None, None, _vp(st),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()               # the launch returned: the stream drains
    assert int(st.item()) == -8            # PHS_ETIMEOUT
    assert torch.equal(out[1:], ref[1:])   # requests not on the failed warp: unchanged
    again = phs.attn_decode_full_paged(q, pool, dev(bt), dev(lens), ms, out_dtype=torch.float32)
    torch.cuda.synchronize()               # the context is still usable
    assert torch.equal(again, ref)


@pytest.mark.parametrize("B", [4, 80])  # 8 units: one CTA each; 160 units: persistent warps
def test_swa_kernel_wait_runs_out_and_returns(wait_lib, B):
    Hq, Hkv, D, W = 16, 2, 128, 128
    ring = phs.RingPool(synth.normal_bf16((B, Hkv, W, D), 9, device="cuda"),
                        synth.normal_bf16((B, Hkv, W, D), 10, device="cuda"))
    q = synth.normal_bf16((B, Hq, D), 11, device="cuda")
    rng = np.random.default_rng(B)
    pos = np.concatenate([[3, 127, 64, 0], rng.integers(0, W, B - 4)]).astype(np.int32)
    lens = np.concatenate([[500, 90, 128, 7000], rng.integers(1, 3 * W, B - 4)]).astype(np.int32)
    rp, sl = dev(pos), dev(lens)
    ref = phs.attn_decode_swa_ring(q, ring, rp, sl, out_dtype=torch.float32)
    out = torch.zeros_like(ref)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc_ = ring.c()
    rc = wait_lib.phs_attn_decode_swa_ring(
        _vp(q), Hq, ctypes.byref(rc_), None, _vp(rp), _vp(sl), B, 1 / np.sqrt(D), _vp(out), 1,
        _vp(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == -8
    G = Hq // Hkv
    assert torch.equal(out[0, G:], ref[0, G:])   # request 0's other KV head
    assert torch.equal(out[1:], ref[1:])
    again = phs.attn_decode_swa_ring(q, ring, rp, sl, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(again, ref)
