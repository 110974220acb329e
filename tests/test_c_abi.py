"""The C ABI from plain C: tests/c/plan_from_c.c is compiled as C99 against include/msa.h
(gcc -Werror) and linked to libmsa.so, then run.  It plans a layout through the host-only
entry points.  Its plan must equal the Python binding's plan of the same arrays and the
oracle's canonical plan; its useful-FLOP count must equal the closed form.  No GPU is used."""
import os
import subprocess

import numpy as np
import pytest

import segmented_kv_attention_msa_b300 as msa
from segmented_kv_attention_msa_b300 import build as B
from segmented_kv_attention_msa_b300 import workload as W
from oracle import msa_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    B.build()
    exe = str(tmp_path_factory.mktemp("c_abi") / "plan_from_c")
    pkg = os.path.dirname(msa.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC,
           os.path.join(ROOT, "tests", "c", "plan_from_c.c"), msa.LIB_PATH, "-Wl,-rpath," + pkg, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    out = {}
    for line in r.stdout.splitlines():
        key, _, rest = line.partition(" ")
        out[key] = rest.split()
    return out


def layout():
    """The C program's layout as the seeded generator's Layout record."""
    return W.Layout(mode="prefill", num_heads_q=4, num_heads_kv=2, head_dim=64, num_seqs=1, num_pool_blocks=2,
                    block_pos=np.array([16, 0], np.int32), block_fill=np.array([16, 16], np.int32),
                    block_table=np.array([[1, 0]], np.int32), segments=np.array([[0, 0, 2]], np.int32),
                    cu_q=np.array([0, 9], np.int32), q_pos=np.arange(32, 41, dtype=np.int32), qk_std=1.0, v_std=1.0)


def test_c_caller_gets_the_python_and_oracle_plan(c_output):
    assert int(c_output["version"][0]) == int(msa.lib().msa_version())
    ex = np.array([int(x) for x in c_output["export"]], np.int32)
    np.testing.assert_array_equal(ex, msa.Plan.from_layout(layout()).export())
    np.testing.assert_array_equal(ex, O.canonical_plan(layout()))


def test_c_caller_flops_closed_form(c_output):
    # each of the 9 chunk rows sees the 32 pool keys and the chunk rows up to itself
    pairs = 9 * 32 + sum(range(1, 10))
    assert int(c_output["useful_flops"][0]) == 4 * 64 * 4 * pairs
    assert int(c_output["kv_tokens"][0]) == 32 + 9


def test_c_caller_error_path(c_output):
    assert c_output["overlap"] == [str(-3), "null"]   # MSA_ERR_POS_OVERLAP, *out reset
