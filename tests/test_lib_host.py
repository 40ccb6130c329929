"""Host-side checks of the C-ABI library: it loads, exports every function
include/kv_pool.h declares, and its layout gates agree with the oracle's.
No compute call is made (no GPU here)."""
import ctypes

import pytest

import gather_translate_kv_gb300 as gt
import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    from gather_translate_kv_gb300 import build

    build.build()
    return gt.lib()


def test_exports_every_declared_symbol(lib):
    names = gt.header_functions()
    assert len(names) >= 11, names
    for n in names:
        assert hasattr(lib, n), f"libgtkv.so does not export {n}"


def test_device_error_bits_match_the_header():
    """The binding's KV_DEV_ERR_* constants are the header's #defines."""
    import re

    defs = dict(re.findall(r"^#define (KV_DEV_ERR_\w+) (\d+)", open(gt.HEADER).read(), flags=re.M))
    assert set(defs) == {"KV_DEV_ERR_ROW", "KV_DEV_ERR_V2P", "KV_DEV_ERR_TABLE", "KV_DEV_ERR_FORM",
                         "KV_DEV_ERR_TIMEOUT"}
    for name, value in defs.items():
        assert getattr(gt, name) == int(value), name


def test_status_strings(lib):
    for code, name in gt.STATUS.items():
        assert gt.kv_status_string(code) == name


def test_required_bytes_match_layout_table(lib):
    for r in oracle_pins._rows(oracle_pins.os.path.join(oracle_pins.GOLDEN, "layout_table.txt")):
        L, H, D, it, ps, P = map(int, r[:6])
        R, pb, tot, tp, nr, lve = map(int, r[7:])
        total, pad = gt.kv_pool_required_bytes(gt.make_desc(L, H, D, it, ps, P))
        assert (total, pad) == (tot, tp)


# (desc kwargs, expected library code, expected oracle verdict)
GATES = [
    (dict(layer_num=2, head_num=2, head_dim=8, itemsize=2, page_size=4, num_pages=64), 0, "ok"),
    (dict(layer_num=2, head_num=2, head_dim=8, itemsize=2, page_size=4, num_pages=64, v_head_dim=16), -2,
     "asymmetric"),
    (dict(layer_num=80, head_num=1, head_dim=64, itemsize=1, page_size=256, num_pages=52428), 0, "ok"),
    (dict(layer_num=80, head_num=1, head_dim=64, itemsize=1, page_size=256, num_pages=52429), -3, "id_bound"),
    (dict(layer_num=1, head_num=1, head_dim=16, itemsize=1, page_size=2, num_pages=1 << 29), -3, "id_bound"),
    (dict(layer_num=1, head_num=1, head_dim=16, itemsize=1, page_size=2, num_pages=(1 << 29) - 1), 0, "ok"),
    (dict(layer_num=2, head_num=2, head_dim=8, itemsize=2, page_size=4, num_pages=64, anchor_bytes=3), -5,
     "anchor"),
    (dict(layer_num=2, head_num=0, head_dim=8, itemsize=2, page_size=4, num_pages=64), -1, "bad_arg"),
    (dict(layer_num=2, head_num=2, head_dim=8, itemsize=2, page_size=0, num_pages=64), -1, "bad_arg"),
    # MLA: one latent row per layer, asymmetric head dims admitted, bound over L blocks
    (dict(layer_num=2, head_num=1, head_dim=16, itemsize=2, page_size=4, num_pages=64, v_head_dim=128,
          latent_only=True), 0, "ok"),
    (dict(layer_num=61, head_num=1, head_dim=576, itemsize=2, page_size=64, num_pages=550072, latent_only=True), 0,
     "ok"),
    (dict(layer_num=61, head_num=1, head_dim=576, itemsize=2, page_size=64, num_pages=550073, latent_only=True), -3,
     "id_bound"),
]


@pytest.mark.parametrize("kw,code,verdict", GATES)
def test_gates_agree_with_oracle(lib, kw, code, verdict):
    d = gt.make_desc(**kw)
    rc = lib.kv_pool_required_bytes(ctypes.byref(d), None, None)
    assert rc == code, gt.STATUS.get(rc)
    g = oracle.Geometry(kw["layer_num"], kw["head_num"], kw["head_dim"], kw["itemsize"], kw["page_size"],
                        kw["num_pages"], kw.get("anchor_bytes", 0), kw.get("v_head_dim"), kw.get("latent_only", False))
    assert oracle.Oracle(g).check() == verdict


def test_alignment_gates(lib):
    # rows that are not a whole number of 16-byte vectors, and a 16-byte anchor rule
    assert lib.kv_pool_required_bytes(ctypes.byref(gt.make_desc(1, 1, 4, 2, 4, 8)), None, None) == -5
    assert lib.kv_pool_required_bytes(ctypes.byref(gt.make_desc(1, 1, 8, 2, 4, 8, anchor_bytes=8)), None,
                                      None) == -5


def test_create_rejects_short_buffer_before_touching_the_device(lib):
    # a fake aligned device pointer: the tail-pad gate is checked on the host
    # before any CUDA call, so nothing is dereferenced
    d = gt.make_desc(2, 2, 8, 2, 4, 64)
    o = oracle.Oracle(oracle.Geometry(2, 2, 8, 2, 4, 64))
    lve = o.sizes()["last_view_end"]
    h = ctypes.c_void_p()
    rc = lib.kv_pool_create(ctypes.byref(d), ctypes.c_void_p(1 << 20), lve - 1, ctypes.byref(h))
    assert rc == -4 and not h.value
    rc = lib.kv_pool_create(ctypes.byref(d), ctypes.c_void_p((1 << 20) + 8), lve, ctypes.byref(h))
    assert rc == -5 and not h.value
    assert lib.kv_pool_create(ctypes.byref(d), None, 0, None) == -1


def test_entry_points_reject_null_pool(lib):
    vp = ctypes.c_void_p
    assert lib.kv_translate(None, vp(16), 1, None, 0, vp(16), None) in (-1, -6)
    assert lib.kv_store_layer(None, 0, vp(16), 1, vp(16), vp(16), None) in (-1, -6)
    assert lib.kv_move(None, vp(16), vp(16), 1, None) in (-1, -6)
    assert lib.kv_pool_destroy(None) == 0


def c_abi_program(tmp_path, with_cuda: bool):
    """Build tests/c_abi_roundtrip.c as a plain C99 program against libgtkv.so."""
    import os
    import subprocess

    from gather_translate_kv_gb300 import build

    lib_path = build.build()
    exe = tmp_path / ("c_abi_gpu" if with_cuda else "c_abi_host")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c_abi_roundtrip.c")
    cuda = "/usr/local/cuda"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", build.INCLUDE, src, "-o", str(exe),
           lib_path, f"-Wl,-rpath,{os.path.dirname(lib_path)}"]
    if with_cuda:
        cmd += ["-DWITH_CUDA", "-I", f"{cuda}/include", f"-L{cuda}/lib64", "-lcudart",
                f"-Wl,-rpath,{cuda}/lib64"]
    subprocess.check_call(cmd)
    return str(exe)


def test_c_abi_from_plain_c(tmp_path):
    """The header compiles as C99 with -Werror, the library links from C, and
    the host-side gates answer as documented (no GPU needed)."""
    import subprocess

    exe = c_abi_program(tmp_path, with_cuda=False)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c abi: ok" in r.stdout


@pytest.mark.gpu
def test_c_abi_round_trip_on_gpu(tmp_path):
    """translate -> store -> gather through the C ABI from a C program."""
    import subprocess

    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")

    exe = c_abi_program(tmp_path, with_cuda=True)
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
