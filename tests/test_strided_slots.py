"""The strided gather's slot arithmetic (P in {3, 5, 6, 7}) against plain
enumeration, on the CPU: a host harness compiled from the library's own
header prints the first owned row of each page and each request's length in
slots.

Partition r owns global tokens t with t mod P = r (sglang pull 33926,
"Decode layout").  Enumerated here: token t sits in page t // 64 at row
t % 64; each page's owned rows are numbered k = 0, 1, ... in row order and
take slot 8 * apg * page + k, with apg = ceil(ceil(64 / P) / 8) atoms of 8
rows per page; a request of length L needs the slots up to and including
that of its last owned token.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def dump():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    out_dir = os.path.join(HERE, "native", "_build")  # git-ignored
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "strided_slots_dump")
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-I",
                    os.path.join(ROOT, "mla_paged_decode_gb300", "csrc"), "-I",
                    os.path.join(ROOT, "include"), os.path.join(HERE, "native", "strided_slots_dump.cu"),
                    "-o", exe], check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    y0, slots = {}, {}
    for line in out.splitlines():
        kind, P, r, x, v = line.split()
        (y0 if kind == "y0" else slots)[(int(P), int(r), int(x))] = int(v)
    return y0, slots


def apg_of(P):
    return (-(-64 // P) + 7) // 8


def enumerate_slots(P, r, L):
    apg = apg_of(P)
    last = None
    for page in range((L + 63) // 64):
        owned_rows = [t % 64 for t in range(64 * page, min(64 * page + 64, L)) if t % P == r]
        if owned_rows:
            last = 8 * apg * page + len(owned_rows) - 1
        assert len([t for t in range(64 * page, 64 * page + 64) if t % P == r]) <= 8 * apg
    return 0 if last is None else last + 1


@pytest.mark.parametrize("P", [3, 5, 6, 7])
def test_first_owned_row_of_each_page(dump, P):
    y0, _ = dump
    for r in range(P):
        for lp in range(3 * P):
            first = min(t % 64 for t in range(64 * lp, 64 * lp + 64) if t % P == r)
            assert y0[(P, r, lp)] == first, (P, r, lp)


@pytest.mark.parametrize("P", [3, 5, 6, 7])
def test_request_length_in_slots(dump, P):
    _, slots = dump
    for r in range(P):
        for L in range(0, 701):
            assert slots[(P, r, L)] == enumerate_slots(P, r, L), (P, r, L)


def test_a_page_never_needs_more_atoms_than_given():
    for P in (3, 5, 6, 7):
        most = max(len([t for t in range(64 * lp, 64 * lp + 64) if t % P == r])
                   for r in range(P) for lp in range(P))
        assert most <= 8 * apg_of(P) and most > 8 * (apg_of(P) - 1), P
