"""Resource checks of the kernels from the compiler's own report
(``nvcc -Xptxas -v``: register, stack and spill counts only). No tensor-core kernel spills
registers or uses a stack frame, except the attention kernel, whose spill is
held to the few bytes the compiler currently places there (a guard against
growth: a larger spill in its sub-tile loop costs time); every instantiation's
registers at launch fit its block on one SM; and each attention instantiation's
``setmaxnreg`` split (control warps down, softmax warps up) adds up to no more
than the registers its block was launched with, since a split above that would
wait forever at ``setmaxnreg.inc``. The fp32 kernels of the two fp32 benchmark
configurations do not spill either. Runs on the CPU: nvcc cross-compiles for
sm_103a without a GPU; the shape constants come from the kernels' own header,
compiled into a small host program."""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

from pair_representation_triangular_gb300 import build as tbuild

TC_SRCS = [os.path.join(tbuild.CSRC, f) for f in ("tc_k1.cu", "tc_k2.cu", "tc_k3.cu")]
REGS_PER_SM = 65536
# Every instantiation the launchers dispatch to: (D, h) for the projection
# kernel, d for the attention kernel, D for the output kernel.
K1_SHAPES = [(32, 1), (32, 2), (64, 1), (64, 2), (64, 4), (128, 2), (128, 4), (128, 8)]
K2_DIMS = [16, 32, 64]
K3_DIMS = [32, 64, 128]


def _ptxas_report(srcs):
    try:
        cc = tbuild.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    kernels = {}
    with tempfile.TemporaryDirectory() as d:
        for src in srcs:
            r = subprocess.run([cc, *tbuild.ARCH, *tbuild.CFLAGS, "-Xptxas", "-v", "-c", src,
                                "-o", os.path.join(d, "k.o")],
                               capture_output=True, text=True, timeout=900)
            assert r.returncode == 0, r.stderr[-2000:]
            cur = None
            for line in (r.stdout + r.stderr).splitlines():
                m = re.search(r"Compiling entry function '([^']+)'", line)
                if m:
                    cur = m.group(1)
                    kernels[cur] = {}
                    continue
                m = re.search(r"Function properties for (\S+)", line)
                if m:
                    # The properties that follow belong to this function, which
                    # is the current entry only if the names agree.
                    if cur is not None and m.group(1) != cur:
                        cur = None
                    continue
                if cur is None:
                    continue
                m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads",
                              line)
                if m:
                    kernels[cur].update(stack=int(m[1]), spill_st=int(m[2]), spill_ld=int(m[3]))
                m = re.search(r"Used (\d+) registers", line)
                if m:
                    kernels[cur]["regs"] = int(m[1])
    return kernels


@pytest.fixture(scope="module")
def report():
    return _ptxas_report(TC_SRCS)


@pytest.fixture(scope="module")
def shapes():
    """kThreads, kRegsCtl, kRegsSoftmax of each attention instantiation, from the
    shape header the kernels are built with."""
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    prog = ('#include <stdio.h>\n#include "tc_shapes.h"\nusing namespace tri_tc;\n'
            'template <int D> void p() { printf("%d %d %d %d\\n", D, k2::Shape<D>::kThreads, '
            'k2::Shape<D>::kRegsCtl, k2::Shape<D>::kRegsSoftmax); }\n'
            'int main() { p<16>(); p<32>(); p<64>(); return 0; }\n')
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "s.cpp"), os.path.join(d, "s")
        with open(src, "w") as f:
            f.write(prog)
        subprocess.run([gxx, "-std=c++17", "-I", tbuild.CSRC, src, "-o", exe], check=True,
                       timeout=120)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return {int(a): (int(b), int(c), int(e)) for a, b, c, e in
            (line.split() for line in out.strip().splitlines())}


def _kernel(report, name, targs):
    """The report of kernel `name` instantiated with integer template arguments
    `targs` (mangled as <length><name>I Li<arg>E ... E)."""
    tag = f"{len(name)}{name}I" + "".join(f"Li{a}E" for a in targs) + "E"
    hits = [v for k, v in report.items() if tag in k]
    assert len(hits) == 1, (tag, list(report))
    return hits[0]


# Spill bytes the compiler places in the attention kernel at present (stores,
# loads, stack frame), measured on this toolkit: none for d = 16; a few bytes
# for d = 64, whose unit epilogue holds 64 accumulator columns, and for d = 32
# since the softmax keeps the unit's sub-tile count in a register (a spill-free
# arrangement that re-read it from shared memory every sub-tile was slower).
# Where they land moves with unrelated code changes (register allocation), so
# the bound is what this guards.
ATTN_SPILL_LIMIT = {16: {"spill_st": 0, "spill_ld": 0, "stack": 0},
                    32: {"spill_st": 4, "spill_ld": 16, "stack": 8},
                    64: {"spill_st": 4, "spill_ld": 12, "stack": 8}}

CASES = ([("ln_proj_tc", s, 576) for s in K1_SHAPES] + [("row_attn_tc", (d,), None) for d in K2_DIMS]
         + [("gate_out_tc", (D,), 320) for D in K3_DIMS])


@pytest.mark.parametrize("name,targs,threads", CASES,
                         ids=[f"{n}<{','.join(map(str, t))}>" for n, t, _ in CASES])
def test_no_spills_and_registers_fit(report, shapes, name, targs, threads):
    k = _kernel(report, name, targs)
    if name == "row_attn_tc":
        threads = shapes[targs[0]][0]
        assert all(k[key] <= lim for key, lim in ATTN_SPILL_LIMIT[targs[0]].items()), k
    else:
        assert k["stack"] == 0 and k["spill_st"] == 0 and k["spill_ld"] == 0, k
    assert k["regs"] * threads <= REGS_PER_SM, k


def test_mask_and_bias_kernels_do_not_spill(report):
    for tag in ("12mask_summaryE", "17mask_summary_colsE", "9bias_rowsE"):
        hits = [v for k, v in report.items() if tag in k]
        assert len(hits) == 1, (tag, list(report))
        k = hits[0]
        assert k["stack"] == 0 and k["spill_st"] == 0 and k["spill_ld"] == 0, (tag, k)


@pytest.mark.parametrize("d", K2_DIMS)
def test_attention_register_split_fits_the_launch(report, shapes, d):
    with open(os.path.join(tbuild.CSRC, "tc_k2.cu")) as f:
        src = f.read()
    # Roles: warps 0-3 (TMA producer, MMA issuers) lower to kRegsCtl, the other
    # warps (the softmax warpgroups) raise to kRegsSoftmax.
    assert re.search(r"if \(warp < 4\) \{\s*tc::regs_dec<kRegsCtl>\(\);", src)
    assert re.search(r"\} else \{\s*//[^\n]*\n\s*tc::regs_inc<kRegsSoftmax>\(\);", src)
    threads, ctl, sm = shapes[d]
    launch = _kernel(report, "row_attn_tc", (d,))["regs"]
    warps = threads // 32
    for n in (ctl, sm):
        assert n % 8 == 0 and 24 <= n <= 256
    assert ctl <= launch <= sm
    assert 32 * (4 * ctl + (warps - 4) * sm) <= launch * threads


F32_SRC = os.path.join(tbuild.CSRC, "kernels_f32.cu")
# fp32 kernels of the two fp32 benchmark configurations (d = 16 and d = 32,
# starting node; d = 32 ending node) and the 128-wide heads, by a unique piece
# of their mangled names.
F32_SPILL_FREE = ("11ln_proj_f32E", "12gate_out_f32E", "row_attn_f32ILi16ELi32ELb0EE",
                  "row_attn_f32ILi32ELi32ELb0EE", "row_attn_f32ILi32ELi32ELb1EE",
                  # d = 128 (two threads per query), both nodes
                  "row_attn_f32ILi128ELi16ELb0EE", "row_attn_f32ILi128ELi16ELb1EE")


def test_fp32_benchmark_kernels_do_not_spill():
    try:
        cc = tbuild.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        r = subprocess.run([cc, *tbuild.ARCH, *tbuild.CFLAGS, "-Xptxas", "-v", "-c", F32_SRC,
                            "-o", os.path.join(d, "k.o")],
                           capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    spills, cur = {}, None
    for line in (r.stdout + r.stderr).splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur:
            spills[cur] = int(m[1]) + int(m[2])
    for key in F32_SPILL_FREE:
        hits = [v for k, v in spills.items() if key in k]
        assert len(hits) == 1, (key, list(spills))
        assert hits[0] == 0, (key, hits[0])
