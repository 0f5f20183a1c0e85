"""Host-side checks of the C ABI that need no GPU.

* the library loads and exports every function include/mt_sgemm.h declares;
* the library's padding rule, vector rule and staged layout agree with the
  oracle's restatement of the pages (oracle/smem_rules.py), which is pinned
  to the pages' worked examples in test_oracle_pins.py;
* the tile plans the library would launch keep every shared-memory access
  conflict-free under the oracle's bank simulator, and the unpadded plans
  show the conflict the rule removes;
* argument errors, aliasing and the shared-memory budget are rejected on the
  host before anything is launched; without a GPU the computing entry points
  report MT_ERR_NO_DEVICE, and without the library the binding raises
  (there is no CPU fallback); no source of the package names the oracle.
"""
import ctypes
import os
import re
import subprocess
import sys

import pytest

import tiled_fp32_gemm_gb300 as mt
from tiled_fp32_gemm_gb300 import build as mt_build
from oracle import smem_rules as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HAS_GPU = False
try:
    import torch
    HAS_GPU = torch.cuda.is_available()
except Exception:  # pragma: no cover
    pass


@pytest.fixture(scope="module", autouse=True)
def built_library():
    assert mt_build.build() == mt.LIB_PATH
    return mt.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(mt_\w+)\s*\(", text))
    return names


def test_every_declared_function_is_exported_and_bound():
    names = declared_functions()
    assert names, "no declarations found"
    handle = ctypes.CDLL(mt.LIB_PATH)
    for n in sorted(names):
        assert hasattr(handle, n), f"{n} not exported"
    assert names == set(mt.SIGNATURES), "binding and header disagree"
    assert mt.mt_version() >= 100
    assert mt.mt_status_string(mt.MT_ERR_SMEM_BUDGET) == "shared-memory budget exceeded"


def test_checked_build_exports_the_same_entry_points_and_says_so():
    """The bounds-checked variant has the whole C ABI; its mt_bounds_status
    answers (no device here: MT_ERR_NO_DEVICE), while the normal build
    reports that it checks nothing."""
    assert mt_build.build(checked=True) == mt.CHECKED_LIB_PATH
    handle = mt.checked_lib()
    for n in sorted(declared_functions()):
        assert hasattr(handle, n), f"{n} not exported by the checked build"
    out = ctypes.c_int64(-7)
    site = ctypes.c_int(-7)
    st = mt.lib().mt_bounds_status(ctypes.byref(out), ctypes.byref(site), None, None)
    assert st == mt.MT_ERR_UNSUPPORTED and out.value == -7 and site.value == -7
    st = handle.mt_bounds_status(ctypes.byref(out), ctypes.byref(site), None, None)
    assert st == (mt.MT_OK if HAS_GPU else mt.MT_ERR_NO_DEVICE)


C_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include "mt_sgemm.h"

int main(void) {
    mt_smem_layout l;
    mt_plan p;
    mt_config c = {0};
    if (mt_smem_row_padding(16, 4) != 1 || mt_smem_row_padding(16, 2) != 0) return 1;
    if (mt_smem_layout_make(4, 16, 1, 2, &l) != MT_OK || l.row_stride != 17) return 2;
    if (mt_smem_layout_offset(&l, 1, 2, 3) != 1 * 68 + 2 * 17 + 3) return 3;
    c.variant = MT_VARIANT_P18;
    if (mt_sgemm_plan(NULL, NULL, NULL, 100, 72, 80, &c, 48 * 1024, &p) != MT_OK) return 4;
    if (p.bm != 4 || p.bn != 8 || p.bk != 16 || p.pad_a != 1) return 5;
    if (mt_sgemm_plan(NULL, NULL, NULL, -1, 4, 4, NULL, 48 * 1024, &p) != MT_ERR_INVALID_ARG)
        return 6;
    /* Without a GPU the status check reports that, and touches nothing. */
    if (getenv("MT_EXPECT_NO_DEVICE") && mt_check_device_status(0) != MT_ERR_NO_DEVICE)
        return 7;
    printf("%s|%d\n", mt_status_string(MT_ERR_SMEM_BUDGET), mt_version());
    return 0;
}
"""


@pytest.mark.parametrize("checked", [False, True], ids=["normal", "checked"])
def test_header_is_c_and_the_library_links_from_c(tmp_path, checked):
    """A C99 program includes include/mt_sgemm.h, links the library (or its
    bounds-checked build) and calls its host-only entry points (padding
    rule, layout, plan, status names): the boundary works from plain C, no
    C++ or torch involved."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    lib_path = mt_build.build(checked=checked)
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(mt_build.nvcc())), "include")
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    lib_dir = os.path.dirname(lib_path)
    lib_name = os.path.basename(lib_path)[3:-3]  # libX.so -> X
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src), "-o", str(exe), "-L", lib_dir, f"-l{lib_name}",
                        f"-Wl,-rpath,{lib_dir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ)
    if not HAS_GPU:
        env["MT_EXPECT_NO_DEVICE"] = "1"
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0, (r.returncode, r.stderr)
    name, version = r.stdout.strip().split("|")
    assert name == "shared-memory budget exceeded" and int(version) == mt.mt_version()


def test_binding_refuses_host_tensors():
    """The torch wrappers hand only CUDA tensors to the library: a host
    tensor is refused before any call (there is no CPU path)."""
    import torch
    a = torch.zeros(4, 3)
    b = torch.zeros(3, 5)
    for call in (lambda: mt.sgemm(a, b), lambda: mt.gemm(a, b),
                 lambda: mt.gemm_mixed(a.to(torch.bfloat16), b.to(torch.bfloat16))):
        with pytest.raises(TypeError):
            call()


def test_padding_rule_matches_pages_and_oracle():
    for c in (1, 2, 3, 4, 5, 7, 8, 12, 16, 17, 24, 31, 32, 33, 48, 64, 96, 128):
        for r in range(1, 33):
            assert mt.mt_smem_row_padding(c, r) == R.row_padding(c, r), (c, r)
    assert mt.mt_smem_row_padding(0, 4) == -1
    assert mt.mt_smem_row_padding(16, 0) == -1


def test_vector_rule_matches_oracle():
    for c in range(4, 260, 4):
        for r in range(1, 9):
            assert mt.mt_smem_vector_row_padding(c, r) == R.vector_row_padding(c, r)
    assert mt.mt_smem_vector_row_padding(6, 2) == -1


def test_layout_matches_oracle():
    for rows, cols, pad, stages in [(4, 16, 1, 2), (16, 8, 0, 2), (128, 32, 4, 3),
                                    (32, 128, 0, 4), (1, 1, 0, 1), (7, 5, 3, 5)]:
        st, L = mt.mt_smem_layout_make(rows, cols, pad, stages)
        assert st == mt.MT_OK
        ref = R.SharedBuffer(rows, cols, pad, stages)
        assert (L.row_stride, L.stage_size, L.size, L.nbytes) == \
            (ref.row_stride, ref.stage_size, ref.size, ref.nbytes)
        for s in range(stages):
            for r in {0, rows - 1, rows // 2}:
                for c in {0, cols - 1, cols // 2}:
                    assert mt.mt_smem_layout_offset(L, s, r, c) == ref.element(s, r, c)
        for bad in [(stages, 0, 0), (0, rows, 0), (0, 0, cols), (-1, 0, 0)]:
            assert mt.mt_smem_layout_offset(L, *bad) == -1
    for bad in [(0, 4, 0, 1), (4, 0, 0, 1), (4, 4, -1, 1), (4, 4, 0, 0)]:
        assert mt.mt_smem_layout_make(*bad)[0] == mt.MT_ERR_INVALID_ARG


GB300_SMEM = 232448  # opt-in dynamic shared memory per block on sm_103


def plan(M, N, K, limit=GB300_SMEM, **kw):
    st, p = mt.mt_sgemm_plan(None, None, None, M, N, K,
                             mt.make_config(**kw) if kw else None, limit)
    return st, p


def ffma_warp_accesses(p):
    """Byte addresses of warp 0's shared reads and cp.async writes, per
    instruction, each with its access width in bytes.

    Lane layout restated from the kernel's description: a warp tile of
    WM x WN, TM x TN outputs per thread, lanes numbered M-fastest.  Row-major
    A (pack_a 0-2): thread (lm, ln) reads A rows i*LM + lm, a float4 of four
    k at a time.  K-major A (pack_a 3-5, tile As[k][m]): it reads rows in
    fours, q*LM*4 + lm*4 .. +3, one float4 per k.  Either way it reads B
    columns g*LN*4 + ln*4.  A K-major tile is filled with 16-byte chunks
    along M (pack_a 3, 5) or gathered with 4-byte copies in 8 x 4 blocks,
    8 lanes along K (pack_a 4).
    """
    WM, WN, TM, TN = p.wm, p.wn, p.tm, p.tn
    LM = WM // TM
    LN = 32 // LM
    kmajor = p.pack_a >= 3
    la = (R.SharedBuffer(p.bk, p.bm, p.pad_a, p.stages) if kmajor
          else R.SharedBuffer(p.bm, p.bk, p.pad_a, p.stages))
    lb = R.SharedBuffer(p.bk, p.bn, p.pad_b, p.stages)
    b_base = la.nbytes
    reads = []
    if kmajor:
        for k in range(p.bk):
            for q in range(TM // 4):
                reads.append(([4 * la.element(0, k, q * LM * 4 + (lane % LM) * 4)
                               for lane in range(32)], 16))
    else:
        for k4 in range(p.bk // 4):
            for i in range(TM):
                reads.append(([4 * la.element(0, i * LM + lane % LM, k4 * 4)
                               for lane in range(32)], 16))
    for k in range(p.bk):
        for g in range(TN // 4):
            reads.append(([b_base + 4 * lb.element(0, k, g * LN * 4 + (lane // LM) * 4)
                           for lane in range(32)], 16))
    writes = []
    if p.pack_a == 4:
        kb, warps = p.bk // 8, p.threads // 32
        m_step = warps // kb * 4
        for t in range(kb * (p.bm // 4) // warps):
            writes.append(([4 * la.element(0, lane % 8, lane // 8 + t * m_step)
                            for lane in range(32)], 4))
    elif kmajor:
        chunks = p.bm // 4
        for t in range(p.bk * chunks // p.threads):
            writes.append(([4 * la.element(0, (tid + t * p.threads) // chunks,
                                           (tid % chunks) * 4) for tid in range(32)], 16))
    else:
        a_chunks = p.bk // 4
        for t in range(p.bm * a_chunks // p.threads):
            writes.append(([4 * la.element(0, (tid + t * p.threads) // a_chunks,
                                           (tid % a_chunks) * 4) for tid in range(32)], 16))
    b_chunks = p.bn // 4
    for t in range(p.bk * b_chunks // p.threads):
        writes.append(([b_base + 4 * lb.element(0, (tid + t * p.threads) // b_chunks,
                                                (tid % b_chunks) * 4) for tid in range(32)], 16))
    return reads, writes


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (1024, 1024, 1024), (128, 256, 64)])
@pytest.mark.parametrize("tile", [dict(), dict(bm=128, bn=256), dict(bm=64, bn=64),
                                  dict(bm=256, bn=128), dict(bm=128, bn=128, wm=32, wn=64),
                                  dict(bm=128, bn=128, wm=64, wn=32)])
def test_ffma_layout_is_conflict_free(shape, tile):
    st, p = plan(*shape, **tile)
    assert st == mt.MT_OK
    reads, writes = ffma_warp_accesses(p)
    for addrs, width in reads + writes:
        assert R.conflict_degree(addrs, width) == 1
    assert p.pad_b == 0  # B is read as a broadcast: the rule gives no padding
    if p.pack_a == 4:
        # Gathered K-major A: 8 k rows are written at the same column at
        # once, so the scalar rule pads by one word, rounded up to a float4.
        assert p.pad_a == -(-R.row_padding(p.bm, 8) // 4) * 4 == 4
    elif p.pack_a in (3, 5):
        # K-major A read one k row at a time: the rule gives no padding.
        assert p.pad_a == R.vector_row_padding(p.bm, 1) == 0


def test_ffma_kmajor_gather_unpadded_would_conflict():
    """The gathered K-major tile without its padding: the 8 k rows a warp
    writes at one column fall in one bank (stride 128 words)."""
    st, p = plan(1024, 1024, 1024, pack_a=4)
    assert st == mt.MT_OK and p.pack_a == 4 and p.pad_a == 4
    la = R.SharedBuffer(p.bk, p.bm, 0, p.stages)
    addrs = [4 * la.element(0, lane % 8, lane // 8) for lane in range(32)]
    assert R.conflict_degree(addrs, 4) == 8


def test_tensor_core_epilogue_square_is_conflict_free():
    """The tensor-core epilogue's staging square (tcgen05.cuh): lane l
    writes row l of a 32 x 32 chunk one element at a time, then reads
    column l one row at a time.  With the row stride the kernels use both
    patterns hit 32 banks; with 32 words (no padding) the row-wise writes
    would all fall in one bank, as the pages' rule predicts for 32 rows
    read at one column."""
    text = open(os.path.join(ROOT, "tiled_fp32_gemm_gb300", "csrc", "tcgen05.cuh")).read()
    stride = int(re.search(r"constexpr int EPI_STRIDE = (\d+);", text).group(1))
    assert stride == 32 + R.row_padding(32, 32)

    def writes(st, i):
        return [4 * (lane * st + i) for lane in range(32)]

    def reads(st, r):
        return [4 * (r * st + lane) for lane in range(32)]

    for k in range(32):
        assert R.conflict_degree(writes(stride, k), 4) == 1
        assert R.conflict_degree(reads(stride, k), 4) == 1
        assert R.conflict_degree(writes(32, k), 4) == 32
        assert R.conflict_degree(reads(32, k), 4) == 1


@pytest.mark.parametrize("shape,trans_a,want", [
    ((4096, 4096, 4096), False, 5),   # large N: transposing copy of A
    ((65536, 128, 4096), False, 4),   # narrow N: gathered inside the kernel
    ((4096, 4096, 4096), True, 3),    # A stored K x M: read as stored
    ((4097, 3001, 2053), True, 5),    # A stored K x M, M % 4 != 0: copy
    ((100, 72, 80), False, 4),
    ((1024, 1024, 1024), False, 5),   # N = 1024, 2^30 multiply-adds: copy
    ((1024, 1023, 1024), False, 4),   # just under: gathered
    ((32768, 4096, 32768), False, 4),  # A^T would need 4 GiB: gathered instead
    ((32768, 4096, 32768), True, 3),   # A stored K x M, readable: as stored
])
def test_ffma_kmajor_source_choice(shape, trans_a, want):
    M, N, K = shape
    st, p = mt.mt_sgemm_general_plan(int(trans_a), 0, M, N, K, None, M if trans_a else K,
                                     None, N, None, N, None, GB300_SMEM)
    assert st == mt.MT_OK and p.pack_a == want, p.pack_a
    assert p.wm and p.tm % 4 == 0


@pytest.mark.parametrize("warp", [dict(wm=64, wn=64), dict(wm=32, wn=64)])
def test_ffma_unpadded_layout_conflicts(warp):
    st, p = plan(4096, 4096, 4096, bm=128, bn=128, bk=32, stages=3, no_pad=True, fma=2, **warp)
    assert st == mt.MT_OK and p.pad_a == 0
    reads, _ = ffma_warp_accesses(p)
    assert max(R.conflict_degree(a, w) for a, w in reads) > 1
    st, q = plan(4096, 4096, 4096, bm=128, bn=128, bk=32, stages=3, fma=2, pack_a=1, **warp)
    rows_per_phase = min(q.wm // q.tm, 8)
    assert q.pad_a == R.vector_row_padding(32, rows_per_phase) == 4


def test_default_variant_from_the_environment(monkeypatch):
    """Calls without a configuration take MT_SGEMM_VARIANT's variant; a
    configuration wins; an unknown name is refused before any launch."""
    for name, want in (("", mt.MT_VARIANT_FFMA), ("ffma", mt.MT_VARIANT_FFMA),
                       ("tf32x3", mt.MT_VARIANT_TF32X3), ("p18", mt.MT_VARIANT_P18)):
        monkeypatch.setenv("MT_SGEMM_VARIANT", name)
        st, p = plan(300, 200, 100)
        assert st == mt.MT_OK and p.variant == want, name
        st, p = plan(300, 200, 100, variant="ffma", bm=128, bn=128)
        assert st == mt.MT_OK and p.variant == mt.MT_VARIANT_FFMA
    monkeypatch.setenv("MT_SGEMM_VARIANT", "cublas")
    assert plan(300, 200, 100)[0] == mt.MT_ERR_INVALID_ARG
    monkeypatch.delenv("MT_SGEMM_VARIANT")
    assert plan(300, 200, 100)[1].variant == mt.MT_VARIANT_FFMA


def test_p18_plan_follows_the_pages():
    st, p = plan(100, 72, 80, variant="p18")
    assert st == mt.MT_OK
    assert (p.bm, p.bn, p.bk, p.stages, p.threads) == (4, 8, 16, 2, 32)
    assert p.pad_a == R.row_padding(16, 4) == 1 and p.pad_b == 0
    assert p.grid == 25 * 9
    # Four output rows read A at the same k: stride 17 is conflict-free,
    # stride 16 is the 2-way conflict of the pages' example.
    for pad, expect in ((1, 1), (0, 2)):
        la = R.SharedBuffer(4, 16, pad, 2)
        addrs = [4 * la.element(0, lane // 8, 5) for lane in range(32)]
        assert R.conflict_degree(addrs, 4) == expect
    st, p = plan(100, 72, 80, variant="p18", no_pad=True)
    assert p.pad_a == 0
    # The single-stage form the page falls back to (two barriers per tile).
    st, p = plan(100, 72, 80, variant="p18", stages=1)
    assert st == mt.MT_OK and p.stages == 1 and p.pad_a == 1
    assert plan(100, 72, 80, variant="p18", stages=3)[0] == mt.MT_ERR_UNSUPPORTED


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_ffma_pipeline_depth_plans(stages):
    """The 128 x 128 x 16 tile at every K-pipeline depth: the same tile and
    padding, shared memory growing with the stage count by the pages'
    formula (stages * rows * (cols + pad) * 4 for A and for B)."""
    st, p = plan(4096, 4096, 4096, bm=128, bn=128, bk=16, wm=64, stages=stages)
    assert st == mt.MT_OK
    assert (p.bm, p.bn, p.bk, p.stages, p.wm, p.tm, p.tn) == (128, 128, 16, stages, 64, 8, 16)
    assert p.pack_a == 5 and p.pad_a == 0 and p.pad_b == 0
    assert p.smem_bytes == (R.SharedBuffer(p.bk, p.bm, p.pad_a, stages).nbytes +
                            R.SharedBuffer(p.bk, p.bn, p.pad_b, stages).nbytes) == \
        stages * 16 * 256 * 4
    reads, writes = ffma_warp_accesses(p)
    for addrs, width in reads + writes:
        assert R.conflict_degree(addrs, width) == 1


def test_budget_is_checked_before_launch():
    # 48 KiB is the pages' conservative budget: the default tile needs more.
    st, p = plan(4096, 4096, 4096, limit=48 * 1024)
    assert st == mt.MT_ERR_SMEM_BUDGET
    assert p.smem_bytes > 48 * 1024
    # Bytes are the staged layouts' sizes: stages * rows * (cols + pad) * 4.
    st, p = plan(4096, 4096, 4096)
    assert p.smem_bytes == (R.SharedBuffer(p.bm, p.bk, p.pad_a, p.stages).nbytes +
                            R.SharedBuffer(p.bk, p.bn, p.pad_b, p.stages).nbytes)
    assert mt.mt_sgemm_plan(None, None, None, 64, 64, 64, None, p.smem_bytes - 1,
                            )[0] in (mt.MT_OK, mt.MT_ERR_SMEM_BUDGET)


def test_alignment_selects_staging_width():
    rnd = lambda b: (b + 255) // 256 * 256  # noqa: E731
    # Default: A staged K-major from a transposed copy (K x M) for a product
    # this wide, B and C with 16-byte accesses; the last partial wave (1024
    # tiles on 2 x 152 CTA slots leave 112) is split in four K slices.
    p = plan(4096, 4096, 4096)[1]
    assert (p.vec_ab, p.vec_c, p.pack_a, p.split_k) == (1, 1, 5, 4)
    assert p.workspace_bytes == 4096 * 4096 * 4 + 112 * 4 * 128 * 128 * 4
    # Row-major A tiles (pack_a = 2): rows that are not whole float4s are
    # staged as stored with 4-byte copies ...
    p = plan(4097, 3001, 2053, pack_a=2)[1]
    assert (p.vec_ab, p.vec_c, p.pack_a, p.workspace_bytes) == (0, 0, 0, 0)
    # ... or (pack_a = 1) copied into padded rows of whole 128-byte lines,
    # A 4097 x 2080 and B 2053 x 3008, then staged in 16-byte chunks; C has
    # scalar stores (N = 3001).
    p = plan(4097, 3001, 2053, pack_a=1)[1]
    assert (p.vec_ab, p.vec_c, p.pack_a) == (1, 0, 1)
    assert p.workspace_bytes == rnd(4097 * 2080 * 4) + rnd(2053 * 3008 * 4)
    # Automatic: K-major A from a copy (2053 x 4128) and B from a copy with
    # padded rows, on 64 x 128 tiles (too few 128 x 128 tiles for three
    # full waves); 1560 tiles on 3 x 152 CTA slots leave 192 for a last
    # wave, whose K tiles go as stream-K runs to 456 CTAs (two partial
    # slots each); on request the split tail cuts them in four K slices.
    p = plan(4097, 3001, 2053)[1]
    assert (p.vec_ab, p.vec_c, p.pack_a, p.bm, p.bn, p.split_k, p.stream_k) == \
        (1, 0, 5, 64, 128, 1, 456)
    assert p.workspace_bytes == (rnd(2053 * 4128 * 4) + rnd(2053 * 3008 * 4) +
                                 2 * 456 * 64 * 128 * 4)
    p = plan(4097, 3001, 2053, schedule=1)[1]
    assert (p.split_k, p.stream_k) == (4, 0)
    assert p.workspace_bytes == (rnd(2053 * 4128 * 4) + rnd(2053 * 3008 * 4) +
                                 192 * 4 * 64 * 128 * 4)
    # Small products gather K-major A inside the kernel: no copy.
    p = plan(100, 72, 81)[1]
    assert (p.pack_a, p.workspace_bytes, p.vec_ab) == (4, 0, 0)
    st, p = mt.mt_sgemm_plan(4, 16, 32, 64, 64, 64, None, GB300_SMEM)  # 4-byte aligned A
    assert st == mt.MT_OK and p.vec_ab == 0


def test_invalid_arguments_rejected_on_host():
    assert plan(-1, 4, 4)[0] == mt.MT_ERR_INVALID_ARG
    assert plan(4, 4, 2 ** 31)[0] == mt.MT_ERR_INVALID_ARG
    assert plan(64, 64, 64, stages=-1)[0] == mt.MT_ERR_INVALID_ARG
    assert plan(64, 64, 64, bm=96)[0] == mt.MT_ERR_UNSUPPORTED
    assert plan(64, 64, 64, variant=7)[0] == mt.MT_ERR_INVALID_ARG
    # Device entry points check arguments before looking for a device.
    assert mt.mt_sgemm(0, 0, 0, -1, 4, 4, 0) == mt.MT_ERR_INVALID_ARG
    assert mt.mt_sgemm(4096, 8192, 0, 4, 4, 4, 0) == mt.MT_ERR_INVALID_ARG  # C is NULL
    # C overlapping A: rejected as aliasing.
    assert mt.mt_sgemm(1 << 20, 1 << 30, (1 << 20) + 64, 16, 16, 16, 0) == mt.MT_ERR_ALIAS
    # M == 0 or N == 0 is a no-op.
    assert mt.mt_sgemm(0, 0, 0, 0, 16, 16, 0) == mt.MT_OK
    # A bias row overlapping C is aliasing; one not 4-byte aligned is invalid.
    gb = mt.mt_sgemm_general_bias
    assert gb(0, 0, 16, 16, 16, 1.0, 1 << 20, 16, 1 << 30, 16, 0.0, (1 << 34) + 64, 1 << 34, 16,
              0, None) == mt.MT_ERR_ALIAS
    assert gb(0, 0, 16, 16, 16, 1.0, 1 << 20, 16, 1 << 30, 16, 0.0, (1 << 36) + 2, 1 << 34, 16,
              0, None) == mt.MT_ERR_INVALID_ARG


@pytest.mark.skipif(HAS_GPU, reason="checks the no-device path")
def test_no_cpu_fallback_without_gpu():
    assert mt.mt_sgemm(1 << 20, 1 << 30, 1 << 34, 16, 16, 16, 0) == mt.MT_ERR_NO_DEVICE
    import numpy as np
    a = np.ones((4, 4), np.float32)
    c = np.zeros((4, 4), np.float32)
    st = mt.mt_sgemm_host(a.ctypes.data, a.ctypes.data, c.ctypes.data, 4, 4, 4, 0, None)
    assert st == mt.MT_ERR_NO_DEVICE
    assert np.all(c == 0)


def test_missing_library_fails_loudly(tmp_path):
    # No CPU fallback: in a fresh interpreter whose library path names
    # nothing, the first call raises instead of computing, and nothing has
    # imported the oracle.
    code = (
        "import sys\n"
        "import tiled_fp32_gemm_gb300 as mt\n"
        f"mt.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
        "try:\n"
        "    mt.mt_sgemm(0, 0, 0, 4, 4, 4, 0)\n"
        "except RuntimeError as e:\n"
        "    assert 'no CPU fallback' in str(e), e\n"
        "    print('raised')\n"
        "assert not [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.split() == ["raised"], r.stdout + r.stderr


def test_product_sources_never_name_the_oracle():
    # The oracle is test infrastructure: no source of the package or of the
    # exported headers imports, includes or names it.
    dirs = [os.path.join(ROOT, "tiled_fp32_gemm_gb300"), os.path.join(ROOT, "include")]
    seen = 0
    for top in dirs:
        for dirpath, dirnames, files in os.walk(top):
            dirnames[:] = [d for d in dirnames if d not in ("_build", "_build_checked",
                                                            "__pycache__")]
            for fn in files:
                if fn.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                    text = open(os.path.join(dirpath, fn)).read()
                    assert not re.search(r"\boracle\b|ref_gemm|smem_rules", text), fn
                    seen += 1
    assert seen >= 10


def test_split_k_plan():
    # Automatically only the last partial wave is split (112 of 1024 tiles
    # on 304 CTA slots, four slices each); an explicit split applies to every
    # tile; each split tile needs one partial tile per slice (after the 64 MB
    # transposed copy of A); split_k = 1 turns splitting off.
    a_copy = 4096 * 4096 * 4
    st, p = plan(4096, 4096, 4096)
    assert st == mt.MT_OK and (p.bm, p.bn) == (128, 128)
    assert p.split_k == 4 and p.grid == 912 + 112 * 4
    assert p.workspace_bytes == a_copy + 112 * 4 * 128 * 128 * 4
    st, p = plan(4096, 4096, 4096, split_k=2)
    assert p.grid == 1024 * 2 and p.workspace_bytes == a_copy + 1024 * 2 * 128 * 128 * 4
    st, p = plan(4096, 4096, 4096, split_k=3)
    assert p.split_k == 3 and p.grid == 1024 * 3
    st, p = plan(4096, 4096, 4096, split_k=1)
    assert p.split_k == 1 and p.grid == 1024 and p.workspace_bytes == a_copy
    st, p = plan(4096, 4096, 4096, split_k=2, pack_a=2)
    assert p.workspace_bytes == 1024 * 2 * 128 * 128 * 4
    # Fewer tiles than SMs: K is cut so the units fill the SMs, slices of at
    # least 512.  512 x 512 x 4096 (long K, few tiles): 32 tiles of 64 x 128,
    # each CTA with two K groups of 4 warps (256 threads), and 4 slices.
    st, p = plan(512, 512, 4096)
    assert (p.bm, p.bn, p.split_k, p.grid, p.threads) == (64, 128, 4, 128, 256)
    # Short K: 64 x 64 tiles, one K group, no slices of 512.
    st, p = plan(512, 512, 512)
    assert (p.bm, p.bn, p.split_k, p.threads) == (64, 64, 1, 128)
    # A split larger than the K tiles is clamped to one K tile per slice.
    st, p = plan(64, 64, 64, split_k=4)
    assert p.split_k == 2


def test_general_form_argument_checks():
    g = mt.mt_sgemm_general
    # Leading dimensions below the row length are rejected before any device work.
    assert g(0, 0, 8, 8, 8, 1.0, 1 << 20, 7, 1 << 30, 8, 0.0, 1 << 34, 8, 0, None) == \
        mt.MT_ERR_INVALID_ARG                                   # lda < K
    assert g(1, 0, 8, 8, 4, 1.0, 1 << 20, 7, 1 << 30, 8, 0.0, 1 << 34, 8, 0, None) == \
        mt.MT_ERR_INVALID_ARG                                   # transposed A: lda < M
    assert g(0, 1, 8, 8, 9, 1.0, 1 << 20, 9, 1 << 30, 8, 0.0, 1 << 34, 8, 0, None) == \
        mt.MT_ERR_INVALID_ARG                                   # transposed B: ldb < K
    assert g(0, 0, 8, 8, 8, 1.0, 1 << 20, 8, 1 << 30, 8, 0.0, 1 << 34, 7, 0, None) == \
        mt.MT_ERR_INVALID_ARG                                   # ldc < N
    assert g(2, 0, 8, 8, 8, 1.0, 1 << 20, 8, 1 << 30, 8, 0.0, 1 << 34, 8, 0, None) == \
        mt.MT_ERR_INVALID_ARG                                   # trans flag not 0/1
    # C's span (rows of ldc floats) overlapping A's span is aliasing ...
    a, c = 1 << 20, (1 << 20) + 4 * 100
    assert g(0, 0, 4, 4, 4, 1.0, a, 64, 1 << 30, 4, 0.0, c, 4, 0, None) == mt.MT_ERR_ALIAS
    # ... but not when A is never read (alpha == 0).
    st = g(0, 0, 4, 4, 4, 0.0, a, 64, 1 << 30, 4, 0.0, c, 4, 0, None)
    assert st in (mt.MT_OK, mt.MT_ERR_NO_DEVICE)


# --- 16-bit inputs (mt_gemm_mixed*) -------------------------------------------
def plan16(M, N, K, dtype=mt.MT_DTYPE_BF16, ta=0, tb=0, lda=0, ldb=0, ldc=0, a=None, b=None,
           c=None, **kw):
    lda = lda or max(M if ta else K, 1)
    ldb = ldb or max(K if tb else N, 1)
    ldc = ldc or max(N, 1)
    return mt.mt_gemm_mixed_plan(dtype, ta, tb, M, N, K, a, lda, b, ldb, c, ldc,
                                 mt.make_config(**kw) if kw else None, GB300_SMEM)


def test_mixed_plan_tiles_and_tail():
    # Without a GPU the plan assumes 152 SMs: 76 resident clusters of two.
    st, p = plan16(8192, 8192, 8192)
    assert st == mt.MT_OK
    # Automatic: CTA pairs on 256 x 256 tiles (32 x 32 = 1024 tiles >= 76).
    assert (p.variant, p.bm, p.bn, p.bk) == (mt.MT_VARIANT_TC16, 256, 256, 64)
    assert p.threads == 192 and p.grid == 152 and p.vec_ab == 1 and p.vec_c == 1
    # 1024 tiles on 76 clusters leave 36 (at most half): split in 2 K slices.
    assert p.split_k == 2 and p.workspace_bytes == 36 * 2 * 256 * 256 * 4
    assert p.smem_bytes <= GB300_SMEM and p.stages * (128 + 128) * 64 * 2 <= p.smem_bytes
    st, p = plan16(4096, 4096, 4096)
    assert (p.bm, p.split_k) == (256, 2) and p.workspace_bytes == 28 * 2 * 256 * 256 * 4
    st, p = plan16(4096, 4096, 4096, split_k=1)
    assert p.split_k == 1 and p.workspace_bytes == 0
    # One CTA per 128 x 256 tile when asked: 512 tiles on 152 SMs leave 56.
    st, p = plan16(4096, 4096, 4096, bm=128)
    assert (p.bm, p.bn, p.grid, p.stages) == (128, 256, 152, 4)
    assert p.split_k == 2 and p.workspace_bytes == 56 * 2 * 128 * 256 * 4
    # Fewer pair tiles than clusters: single CTAs (1024^3: 16 pair tiles).
    st, p = plan16(1024, 1024, 1024)
    assert p.bm == 128
    # Explicit 128-wide tiles; pairs take only 256-wide tiles.
    st, p = plan16(1024, 1024, 1024, bn=128)
    assert st == mt.MT_OK and (p.bm, p.bn) == (128, 128) and p.stages >= 4
    assert plan16(1024, 1024, 1024, bm=256, bn=128)[0] == mt.MT_ERR_UNSUPPORTED


def test_mixed_plan_repacks_what_tma_cannot_read():
    # Row pitches that are not multiples of 8 elements (16 bytes): both
    # operands get padded copies whose rows are whole 128-byte lines, sized
    # rows x round_up(cols, 64) x 2 bytes.
    st, p = plan16(4097, 3001, 2053)
    assert st == mt.MT_OK and p.vec_ab == 0
    rnd = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert p.workspace_bytes == rnd(4097 * 2112 * 2) + rnd(2053 * 3008 * 2)
    # A 2-byte (not 16-byte) aligned base alone also needs the copy.
    st, p = plan16(256, 256, 256, a=(1 << 20) + 2)
    assert p.vec_ab == 0 and p.workspace_bytes == rnd(256 * 256 * 2)
    st, p = plan16(256, 256, 256, a=1 << 20, b=1 << 24)
    assert p.vec_ab == 1 and p.workspace_bytes == 0


def test_mixed_argument_checks():
    assert plan16(64, 64, 64, dtype=0)[0] == mt.MT_ERR_INVALID_ARG
    assert plan16(64, 64, 64, dtype=3)[0] == mt.MT_ERR_INVALID_ARG
    assert plan16(64, 64, 64, variant="tf32x3")[0] == mt.MT_ERR_UNSUPPORTED
    assert plan16(64, 64, 64, bn=64)[0] == mt.MT_ERR_UNSUPPORTED
    assert plan16(64, 64, 64, bk=32)[0] == mt.MT_ERR_UNSUPPORTED
    assert plan16(64, 64, 64, split_k=2)[0] == mt.MT_ERR_UNSUPPORTED
    assert plan16(64, 64, 64, wm=32)[0] == mt.MT_ERR_UNSUPPORTED
    assert plan16(64, 64, 64, variant="tc16")[0] == mt.MT_OK
    # MT_VARIANT_TC16 needs 16-bit inputs.
    assert plan(64, 64, 64, variant="tc16")[0] == mt.MT_ERR_UNSUPPORTED
    g = mt.mt_gemm_mixed_general
    assert g(2, 0, 0, 8, 8, 8, 1.0, 1 << 20, 7, 1 << 30, 8, 0.0, 1 << 34, 8, 0, None) == \
        mt.MT_ERR_INVALID_ARG                                   # lda < K
    assert g(2, 0, 0, 8, 8, 8, 1.0, (1 << 20) + 1, 8, 1 << 30, 8, 0.0, 1 << 34, 8, 0,
             None) == mt.MT_ERR_INVALID_ARG                     # A not 2-byte aligned
    # Aliasing is judged on 2-byte elements: A spans 8 * 64 * 2 = 1024 bytes.
    a = 1 << 20
    assert g(2, 0, 0, 8, 8, 64, 1.0, a, 64, 1 << 30, 8, 0.0, a + 1020, 8, 0, None) == \
        mt.MT_ERR_ALIAS
    st = g(2, 0, 0, 8, 8, 64, 1.0, a, 64, 1 << 30, 8, 0.0, a + 1024, 8, 0, None)
    assert st in (mt.MT_OK, mt.MT_ERR_NO_DEVICE)
    assert mt.mt_gemm_mixed(5, 0, 0, 0, 4, 4, 4, 0) == mt.MT_ERR_INVALID_ARG
    assert mt.mt_gemm_mixed(mt.MT_DTYPE_F16, 0, 0, 0, 0, 4, 4, 0) == mt.MT_OK  # M == 0


def test_stream_k_plans():
    """The stream-K schedule on the host (no GPU: 152 SMs assumed).  The
    tiles past the last whole wave of resident CTAs are dealt out as runs
    of K tiles, two partial slots per stream-K CTA."""
    rnd = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # FFMA at 4096^3, asked for: 1024 tiles of 128 x 128 on 152 x 2 slots,
    # 912 whole tiles, the other 112 tiles' K tiles over 304 CTAs, after
    # the transposed copy of A.
    st, p = plan(4096, 4096, 4096, schedule=2)
    assert st == mt.MT_OK and (p.bm, p.bn, p.split_k, p.stream_k) == (128, 128, 1, 304)
    assert p.grid == 912 + 304
    assert p.workspace_bytes == 4096 * 4096 * 4 + 2 * 304 * 128 * 128 * 4
    # Automatic on the ragged case's 64 x 128 tiles: 1560 tiles on 152 x 3
    # slots, 1368 whole; the copies of A^T and B have rows of whole 128-byte
    # lines (4128 and 3008 floats).
    st, p = plan(4097, 3001, 2053)
    assert (p.bm, p.bn, p.split_k, p.stream_k, p.grid) == (64, 128, 1, 456, 1368 + 456)
    assert p.workspace_bytes == (rnd(2053 * 4128 * 4) + rnd(2053 * 3008 * 4)
                                 + 2 * 456 * 64 * 128 * 4)
    # The split tail on request, and where the split tail leaves a plan
    # whole, stream-K does too (the same bits as before).
    st, p = plan(4097, 3001, 2053, schedule=1)
    assert (p.split_k, p.stream_k, p.grid) == (4, 0, 1368 + 192 * 4)
    st, p = plan(1024, 1024, 1024)
    assert (p.split_k, p.stream_k, p.grid) == (1, 0, 128)
    # Few K tiles: every CTA takes at least two (4 tiles x 3 K tiles: 6 CTAs).
    st, p = plan(100, 72, 80, schedule=2)
    assert st == mt.MT_OK and (p.bm, p.bn, p.stream_k, p.grid) == (64, 64, 6, 6)
    # split_k = 1 turns it off; an explicit split or the one-warp kernel
    # refuses it; an unknown schedule is an argument error.
    assert plan(4096, 4096, 4096, schedule=2, split_k=1)[1].stream_k == 0
    assert plan(4096, 4096, 4096, schedule=2, split_k=2)[0] == mt.MT_ERR_UNSUPPORTED
    assert plan(1024, 1024, 1024, variant="p18", schedule=2)[0] == mt.MT_ERR_UNSUPPORTED
    # A small grid with long K would take the K-grouped tile; asked for
    # stream-K, the automatic choice keeps one group of warps per tile.
    st, p = plan(512, 512, 4096, schedule=2)
    assert st == mt.MT_OK and p.threads == 128 and p.stream_k > 0
    assert plan(512, 512, 4096, bm=64, bn=128, stages=3, schedule=2)[0] == \
        mt.MT_ERR_UNSUPPORTED
    assert plan(1024, 1024, 1024, schedule=3)[0] == mt.MT_ERR_INVALID_ARG
    # 3xTF32 on CTA pairs at 4096^3: 256 tiles of 256 x 256 on 76 clusters,
    # 228 whole, the other 28 tiles' K tiles over the 76 clusters.
    st, p = plan(4096, 4096, 4096, variant="tf32x3", schedule=2)
    assert st == mt.MT_OK and (p.bm, p.split_k, p.stream_k, p.grid) == (256, 1, 76, 152)
    assert p.workspace_bytes == 2 * 2 * 4096 * 4096 * 4 + 2 * 76 * 256 * 256 * 4
    # 16-bit inputs read in place: the partial slots are the whole workspace.
    st, p = plan16(4096, 4096, 4096, schedule=2)
    assert st == mt.MT_OK and (p.bm, p.stream_k, p.grid) == (256, 76, 152)
    assert p.workspace_bytes == 2 * 76 * 256 * 256 * 4


def test_tensor_core_small_grid_split_plans():
    """Tensor-core grids of fewer tiles than half the resident CTAs cut K
    into slices at least 1024 deep (no GPU: 152 SMs assumed)."""
    st, p = plan16(512, 512, 4096)
    assert st == mt.MT_OK and (p.bm, p.bn, p.split_k, p.grid) == (128, 128, 4, 64)
    assert p.workspace_bytes == 16 * 4 * 128 * 128 * 4  # a partial tile per slice
    st, p = plan16(1024, 1024, 1024)  # slices of 512 would not repay the reduce
    assert (p.split_k, p.grid) == (1, 64)
    st, p = plan(512, 512, 4096, variant="tf32x3")
    assert st == mt.MT_OK and (p.bm, p.bn, p.split_k, p.grid) == (128, 64, 4, 128)
    st, p = plan(512, 512, 4096, variant="tf32x3", split_k=1)
    assert (p.split_k, p.grid) == (1, 32)
