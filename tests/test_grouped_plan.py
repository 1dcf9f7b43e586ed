"""Launch plan of the row-group split-row softmax (csrc/grouped_plan.h), on
the CPU: the header is compiled with the host compiler into a small driver
(tests/native/grouped_plan_check.cpp) and its plans are checked against the
invariants the kernel relies on (whole rows per wave of the grid, slices that
fit the registers and the ring, every CTA slot used when rows allow) and
against the plan of the benchmark workload."""
import itertools
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "row_wise_reduction_gb300", "csrc")
DRIVER = os.path.join(ROOT, "tests", "native", "grouped_plan_check.cpp")

MAX_VPT, MAX_SLOTS, MAX_BUFFERS = 7, 160, 8
SMS = 152
OPTIN = 232448  # bytes of dynamic shared memory a CTA may opt in to on GB300


def ring_bytes(per_sm):
    """A CTA's share of the SM's shared memory, as the launcher computes it."""
    return (OPTIN + 1024) // per_sm - 1024 - 256 - 512


def slots_per_row(nvec, vec):
    return (nvec * vec + 255) // 256 + 2


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("plan") / "grouped_plan_check")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC, DRIVER, "-o", exe], check=True)

    def run(cases):
        """cases: (M, nvec, sms, block, per_sm, ring, min_buffers, slots) -> (n, slot_vecs, nbuf, grid)."""
        text = "".join(" ".join(str(v) for v in c) + "\n" for c in cases)
        out = subprocess.run([exe], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
        return [tuple(int(v) for v in line.split()) for line in out if line.strip()]

    return run


def test_benchmark_workload_plan(plan):
    """64 x 2^20 fp32 (262144 vectors a row): 76 CTAs a row (54 KB slices,
    within 512 x 7 vectors), 4 ring buffers, 2 rows per wave over all 152
    SMs; bf16 (131072 vectors): 38 CTAs a row, 4 rows per wave."""
    f32 = (64, 262144, SMS, 512, 1, ring_bytes(1), 2, slots_per_row(262144, 4))
    bf16 = (64, 131072, SMS, 512, 1, ring_bytes(1), 2, slots_per_row(131072, 8))
    assert plan([f32, bf16]) == [(76, 3456, 4, 152), (38, 3456, 4, 152)]


def test_few_rows_widen_the_groups(plan):
    """One 2^20-entry fp32 row spreads over every SM; three rows over 76 CTAs
    each (two rows per wave); a 16 MiB row does not fit 160 CTAs."""
    cases = [(1, 262144, SMS, 512, 1, ring_bytes(1), 2, slots_per_row(262144, 4)),
             (3, 262144, SMS, 512, 1, ring_bytes(1), 2, slots_per_row(262144, 4)),
             (4, 1048576, SMS, 512, 1, ring_bytes(1), 2, slots_per_row(1048576, 4))]
    got = plan(cases)
    assert got[0][0] == 152 and got[0][3] == 152
    assert got[1][0] == 76 and got[1][3] == 152
    assert got[2][0] == 0


def _divisors(k):
    return [d for d in range(1, k + 1) if k % d == 0]


@pytest.mark.parametrize("block,per_sm", [(512, 1), (256, 2)])
def test_plan_invariants(plan, block, per_sm):
    Ms = [1, 2, 3, 5, 19, 36, 64, 155, 512, 4096]
    nvecs = [1000, 2048, 10000, 32768, 65536, 131072, 262144, 375000, 524288, 1048576]
    ring = ring_bytes(per_sm)
    cases = [(M, nv, SMS, block, per_sm, ring, mb, slots_per_row(nv, 4))
             for M, nv, mb in itertools.product(Ms, nvecs, [2, 3, 4])]
    ctas = SMS * per_sm
    for case, (n, slot_vecs, nbuf, grid) in zip(cases, plan(cases)):
        M, nvec, _, _, _, _, min_buffers, slots = case
        width = -(-nvec // n) if n else 0
        fits = [d for d in _divisors(ctas)
                if -(-nvec // d) <= block * MAX_VPT and (-(-nvec // d) + 7) // 8 * 8 * 16 * min_buffers <= ring]
        if n == 0:
            # unsupported: nothing fits, or the group (widened for few rows)
            # would be too large or its slices too small
            if fits:
                k = fits[0]
                while M * k < ctas and k < ctas:
                    k = min(d for d in _divisors(ctas) if d > k)
                assert k > MAX_SLOTS or k > slots or nvec < 32 * k, case
            continue
        assert ctas % n == 0 and n <= MAX_SLOTS and n <= slots, case
        assert width <= block * MAX_VPT and nvec >= 32 * n, case
        assert slot_vecs % 8 == 0 and slot_vecs >= width, case
        assert min_buffers <= nbuf <= MAX_BUFFERS and nbuf * slot_vecs * 16 <= ring, case
        assert grid % n == 0 and 1 <= grid // n <= M and grid <= ctas, case
        # the smallest fitting divisor, raised only while the rows would leave CTA slots idle
        assert n >= fits[0], case
        if M * fits[0] >= ctas:
            assert n == fits[0], case
        else:
            assert M * n >= ctas or n == ctas, case
        if M >= ctas // n:
            assert grid == (ctas // n) * n, case


def test_plans_fit_the_workspace_the_library_asks_for(plan):
    """The row-group form stores its header (256 bytes) and M * n 8-byte slots
    in the caller's workspace: for every plan that applies, that fits in
    rowops_online_softmax_workspace_bytes(M, N) (a host-only query)."""
    from row_wise_reduction_gb300 import build
    from row_wise_reduction_gb300.rowops import library

    build.build()
    q = library().rowops_online_softmax_workspace_bytes
    F32, BF16 = 0, 1
    cases, shapes = [], []
    for M in [1, 3, 36, 64, 155, 4096]:
        for N in [65536, 1 << 18, 1 << 20, 1500000, 1 << 21]:
            for code, vec in [(F32, 4), (BF16, 8)]:
                if N % vec:
                    continue
                for block, per_sm in [(512, 1), (256, 2)]:
                    cases.append((M, N // vec, SMS, block, per_sm, ring_bytes(per_sm), 2, slots_per_row(N // vec, vec)))
                    shapes.append((M, N, code))
    checked = 0
    for (M, N, code), (n, _, _, _) in zip(shapes, plan(cases)):
        if n == 0:
            continue
        assert 256 + M * n * 8 <= q(M, N, code), (M, N, code, n)
        checked += 1
    assert checked > 50
