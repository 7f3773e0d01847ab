"""The C ABI from plain C: tests/abi_client.c is compiled with gcc -std=c11
-Wall -Wextra -Werror -pedantic against include/kivi.h alone and linked to the
built library; its host-only checks must print the expected values. No GPU
call is made (every decode and flush call here fails its checks first)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    from kivi_kv_cache_gb300 import build
    lib = build.build()
    out = str(tmp_path_factory.mktemp("abi") / "abi_client")
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_client.c"),
                    "-o", out, "-L", libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir],
                   check=True)
    r = subprocess.run([out], check=True, capture_output=True, text=True, timeout=120)
    return dict(ln.split(" ", 1) for ln in r.stdout.strip().splitlines())


def test_c_client_host_calls(client):
    assert int(client["version"]) >= 100
    assert client["status_ok"] == "KIVI_OK"
    assert client["status_unsupported"] == "KIVI_ERR_UNSUPPORTED"
    assert (client["flush_559"], client["flush_2059"], client["flush_8209"]) == ("512", "2016", "8160")
    assert client["flush_all_ragged"] == "77"
    assert client["flush_bad"] == "-1"


def test_c_client_argument_checks(client):
    assert int(client["flush_bad_bits"]) == UNSUPPORTED
    assert int(client["flush_bad_dim"]) == UNSUPPORTED
    assert int(client["flush_null_x"]) == INVALID
    assert client["flush_nothing"] == "%d 0" % OK
    assert int(client["dequant_empty"]) == OK
    assert int(client["residual_bad_dim"]) == UNSUPPORTED
    assert client["workspace_qwen8b_positive"] == "1"
    assert client["workspace_one_tile"] == "0"
    assert int(client["decode_no_workspace"]) == WORKSPACE
    assert int(client["decode_bad_group"]) == INVALID
    assert int(client["decode_too_many_heads"]) == UNSUPPORTED
    assert int(client["workspace_init_null"]) == INVALID


def test_c_client_cache(client):
    """The kivi_cache struct has the same layout in C and in the Python
    binding, and its calls check before launching."""
    import ctypes
    import kivi_kv_cache_gb300 as kv
    S = kv._CacheStruct
    assert [int(x) for x in client["cache_layout"].split()] == [
        ctypes.sizeof(S), S.kcodes.offset, S.S_q.offset, S.store_written.offset, S.res_off.offset]
    assert client["cache_prefill_nothing"] == "%d 0" % OK
    assert client["cache_window_past_end"] == "%d 61 100" % INVALID  # rows 100 .. 160 past a 160-row window
    assert int(client["cache_decode_bad_batch"]) == INVALID           # B * Hkv != BH


def test_c_client_plan_info(client):
    # the qwen8b decode (2080 packed + 158 fp16 tokens = 65 + 10 tiles per KV
    # head) takes the warp-pair kernel, planned for 152 SMs without a device;
    # with fp16 scales it takes the one-warp-per-tile kernel
    st, pair, n_split, n_tiles = (int(x) for x in client["plan_qwen8b"].split())
    assert (st, pair, n_tiles) == (OK, 1, 75) and n_split > 1
    assert client["plan_qwen8b_f16s"] == "%d 0" % OK
