"""The C ABI from plain C: tests/c_client/host_client.c is compiled with gcc
against include/pagedkv.h, linked to libpagedkv.so and run (host page-table
calls only, no GPU). Its report must equal the same scenario run through the
oracle's page table (chapter 15's bookkeeping)."""

import os
import shutil
import subprocess

import pytest

from libbuild import ROOT, ensure_built
from oracle.pagetable import PageTable


def oracle_report():
    pt = PageTable(8, 4)  # free list 7 .. 0: page 0 first
    lines = []

    def append(rid, count):
        outs = [pt.append(rid) for _ in range(count)]
        lines.append(f"append {rid}: " + " ".join(str(o["slot"]) for o in outs))
        lines.extend(f"cow {o['cow'][0]} {o['cow'][1]}" for o in outs if o["cow"])

    pt.new(0)
    append(0, 10)
    pt.new(1)
    append(1, 5)
    pt.fork(0, 2)
    append(2, 1)
    lines.append(f"trim 0: {len(pt.trim(0, 6))} released")
    append(0, 1)
    for r in range(3):
        lines.append(f"row {r} len {pt.length[r]}: " + " ".join(str(p) for p in pt.block_row(r)))
    lines.append("free: " + " ".join(str(p) for p in pt.free))
    lines.append("ref: " + " ".join(str(c) for c in pt.ref))
    lines.append(f"used {pt.used()}")
    return lines


def test_c_client_matches_the_oracle(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("needs gcc")
    kb = ensure_built()
    libdir = os.path.dirname(kb.LIB_PATH)
    exe = str(tmp_path / "host_client")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_client", "host_client.c"), "-L", libdir, "-lpagedkv",
                    f"-Wl,-rpath,{libdir}", "-o", exe], check=True, capture_output=True, text=True)
    got = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout.splitlines()
    assert got == oracle_report()
