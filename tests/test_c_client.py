"""The boundary from C: tests/abi_client.c, compiled as strict C99 against
include/demo.h and linked against the library, runs its host-only calls and
prints the results, which are checked here against the oracle's payload sizes
and the conventions the header states.  No kernel is launched.
"""

import os
import shutil
import subprocess

import pytest

import oracle.demo_ref as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "abi_client.c")

EINVAL, ENODEV, ENOTINIT = -1, -3, -5


@pytest.fixture(scope="module")
def client_output():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from decoupled_momentum_optimizer_gb300 import build

    pkg = os.path.dirname(build.build())
    out_dir = os.path.join(ROOT, "_build")  # git-ignored build folder inside the repository
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "abi_client")
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), SRC,
           "-o", exe, "-L", pkg, "-ldemo_gb300", "-Wl,-rpath," + pkg]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    out = {}
    for line in run.stdout.splitlines():
        key, *rest = line.split()
        if key == "status":
            out.setdefault("status", {})[int(rest[0])] = " ".join(rest[1:])
        else:
            out[key] = [int(x) for x in rest]
    return out


def test_header_compiles_as_c99_and_links(client_output):
    assert "init" in client_output


def test_status_names_from_c(client_output):
    st = client_output["status"]
    assert st[0].startswith("DEMO_OK") and st[-1].startswith("DEMO_EINVAL") and st[-6].startswith("DEMO_ENOSPACE")
    assert all(name.startswith("DEMO_") for name in st.values())


@pytest.mark.parametrize("tag,mode,k,step", [("demo_k4", ref.MODE_DEMO, 4, 0), ("random_k8", ref.MODE_RANDOM, 8, 0),
                                             ("stride_k4", ref.MODE_STRIDE, 4, 0),
                                             ("diloco_s6", ref.MODE_DILOCO, 1, 6),
                                             ("diloco_s7", ref.MODE_DILOCO, 1, 7)])
def test_payload_sizes_from_c(client_output, tag, mode, k, step):
    assert tuple(client_output[tag]) == ref.payload_bytes(mode, 32 * 1000, k, step=step, period=8)


def test_payload_size_errors_and_wire_from_c(client_output):
    assert client_output["bad_n"][0] == 0  # n not a multiple of the chunk size
    assert client_output["ternary_k4"][0] == ref.payload_bytes_wire(ref.MODE_DEMO, 32 * 1000, 4,
                                                                     wire=ref.WIRE_TERNARY)[0]


def test_encode_replicas_refusals_from_c(client_output):
    assert client_output["replicas_none"] == [EINVAL]
    assert client_output["replicas_shared_m"] == [EINVAL]


def test_validate_payload_from_c(client_output):
    assert client_output["validate_ok"] == [0]
    assert client_output["validate_dup"] == [EINVAL, 2]
    assert client_output["validate_range"] == [EINVAL, 1]


def test_init_and_fault_word_from_c(client_output):
    init = client_output["init"][0]
    fault_status, fault = client_output["fault"]
    if init == 0:  # a GB300 is present
        assert fault_status == 0 and fault == 0
    else:
        assert init == ENODEV and fault_status == ENOTINIT
