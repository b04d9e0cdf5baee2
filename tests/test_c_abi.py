"""The C ABI from C: a plain C11 client (tests/c_abi_client.c) compiled with
gcc -std=c11 -pedantic against include/lmc.h and linked to liblmc.so runs the
host-side calls (no GPU); its output matches the Python binding and the
values the pages give."""
import os
import shutil
import subprocess

import pytest

import state_cache_paging_gb300 as lmc
import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def client_output(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    out = tmp_path_factory.mktemp("cabi") / "client"
    libdir = os.path.dirname(lmc._lib._name)
    subprocess.run(["gcc", "-std=c11", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(HERE, "c_abi_client.c"), "-o", str(out), f"-L{libdir}", "-llmc",
                    f"-Wl,-rpath,{libdir}"], check=True, capture_output=True, text=True)
    r = subprocess.run([str(out)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.splitlines()
    assert lines[-1] == "done"
    return lines


def _value(lines, key):
    return next(l.split(" ", 1)[1] for l in lines if l.split(" ", 1)[0] == key)


def test_host_rules_from_c(client_output):
    L = client_output
    # Kimi-Linear's N at TP 2 and TP 1 ("Kimi-Linear" recipe table and note)
    assert int(_value(L, "unified_tp2")) == 944
    assert int(_value(L, "unified_tp1")) == 1888
    assert int(_value(L, "negotiate_100_64")) == 128
    assert int(_value(L, "strict_100_64")) == lmc.LMC_ERR_NOT_MULTIPLE
    assert int(_value(L, "negotiate_bad_n")) == lmc.LMC_ERR_INVALID_ARG
    assert int(_value(L, "budget_944_1887")) == lmc.LMC_OK
    assert int(_value(L, "budget_944_1888_joint")) == lmc.LMC_ERR_BUDGET
    assert int(_value(L, "budget_944_1888_separate")) == lmc.LMC_OK
    assert int(_value(L, "store_without_batch")) == lmc.LMC_ERR_INVALID_ARG
    assert int(_value(L, "store_bad_chunk")) == lmc.LMC_ERR_NOT_MULTIPLE
    assert _value(L, "strerror_budget") == lmc.lmc_strerror(lmc.LMC_ERR_BUDGET)
    # racing copies and the mixed-step guard, from C
    assert int(_value(L, "copy_racing")) == lmc.LMC_ERR_OVERLAP
    assert int(_value(L, "copy_fine_null_pool")) == lmc.LMC_ERR_INVALID_ARG
    assert int(_value(L, "copy_without_host_pairs")) == lmc.LMC_ERR_INVALID_ARG
    assert _value(L, "disjoint") == f"{lmc.LMC_OK} -1"
    assert _value(L, "shared") == f"{lmc.LMC_ERR_OVERLAP} 20"


def test_layout_from_c_matches_binding(client_output):
    L = client_output
    cfg = W.CONFIGS[1]
    mem = 1056 * 6 * 2170880
    P = lmc.lmc_layout_build(cfg.layers, cfg.N, cfg.packed, mem)
    assert int(_value(L, "num_kv_groups")) == P.num_kv_groups == 4
    assert int(_value(L, "num_object_groups")) == P.num_object_groups == 2
    assert int(_value(L, "num_slabs")) == P.num_slabs == 6
    assert int(_value(L, "page_size")) == P.page_size == 2170880
    assert int(_value(L, "num_blocks")) == P.num_blocks == 1056
    assert int(_value(L, "pool_bytes")) == P.pool_bytes == mem
    rows = [list(map(int, l.split()[1:])) for l in L if l.startswith("layer ")]
    assert len(rows) == 24
    for i, (idx, kind, kv, slot, og, real, page, base, stride) in enumerate(rows):
        assert idx == i
        assert lmc.LMC_LAYER_NAME[kind] == P.kinds[i]
        assert (kv, slot, og, real, page, base, stride) == (P.kv_group[i], P.slot[i], P.object_group[i],
                                                          P.real_bytes[i], P.page_bytes[i], P.base[i], P.stride[i])
    sizes = {int(l.split()[1]): int(l.split()[2]) for l in L if l.startswith("object_bytes ")}
    assert sizes == {g: P.object_bytes(944, g) for g in range(P.num_object_groups)}
    assert sorted(sizes.values()) == [6 * 1087488, 18 * 2170880]
    assert int(_value(L, "backends_stride_attention")) == P.check_backends(True, False)


def _cuda_home():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime.h")):
            return d
    return None


@pytest.mark.gpu
@pytest.mark.parametrize("cfg_index,ids", [(0, None), (2, [0])])
def test_store_load_from_c_match_oracle(tmp_path, cfg_index, ids):
    """A C11 program (tests/c_abi_gpu_client.c) allocates device memory with
    the CUDA runtime's C API and calls lmc_store / lmc_load through the C ABI
    alone; its arena and reloaded pool equal the oracle's byte for byte."""
    import numpy as np

    import oracle
    cuda = _cuda_home()
    if shutil.which("gcc") is None or cuda is None:
        pytest.skip("gcc or the CUDA toolkit headers not available")
    exe = tmp_path / "gpu_client"
    libdir = os.path.dirname(lmc._lib._name)
    subprocess.run(["gcc", "-std=c11", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c_abi_gpu_client.c"), "-o", str(exe),
                    f"-L{libdir}", "-llmc", f"-L{os.path.join(cuda, 'lib64')}", "-lcudart",
                    f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"],
                   check=True, capture_output=True, text=True)
    import functools
    cfg = W.CONFIGS[cfg_index]
    C = oracle.negotiate_chunk(cfg.requested_chunk, cfg.N)
    inp = W.make_inputs(cfg, functools.partial(oracle.layout, cfg.layers, cfg.N, cfg.packed), C, ids)
    Lo = inp.layout
    cols = max(t.shape[1] for t in inp.tables_src + inp.tables_dst)

    def widen(t):
        out = np.full((t.shape[0], cols), -1, dtype=np.int32)
        out[:, :t.shape[1]] = t
        return out

    d = tmp_path
    with open(d / "case.txt", "w") as f:
        f.write(f"{cfg.N} {int(cfg.packed)} {Lo.pool_bytes} {C} {len(inp.lengths)} {cols} {len(cfg.layers)} "
                f"{Lo.num_kv_groups} {Lo.num_object_groups}\n")
        for l in cfg.layers:
            f.write(f"{lmc.LMC_LAYER[l['kind']]} {int(l.get('token_bytes', 0))} {int(l.get('conv_bytes', 0))} "
                    f"{int(l.get('rec_bytes', 0))} {int(l.get('window', 0))}\n")
        for J in inp.jobs:
            f.write(f"{len(J)}\n")
        f.write(f"{inp.arena_bytes}\n")
    pool_h = W.fill_normal_np(Lo.pool_bytes, 71 + cfg_index)
    pool_h.tofile(d / "pool.bin")
    for k in range(Lo.num_kv_groups):
        widen(inp.tables_src[k]).tofile(d / f"src_{k}.bin")
        widen(inp.tables_dst[k]).tofile(d / f"dst_{k}.bin")
    for g, J in enumerate(inp.jobs):
        np.ascontiguousarray(J, dtype=oracle.JOB_DTYPE).tofile(d / f"jobs_{g}.bin")
    r = subprocess.run([str(exe), str(d)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == "done", r.stdout + r.stderr
    assert int((d / "status.out").read_text()) == 0
    arena_o = np.full(inp.arena_bytes, 0x3C, dtype=np.uint8)
    assert oracle.store(Lo, C, pool_h, inp.tables_src, inp.jobs, arena_o) == 0
    fresh_o = np.full(Lo.pool_bytes, W.SENTINEL, dtype=np.uint8)
    assert oracle.load(Lo, C, fresh_o, inp.tables_dst, inp.jobs, arena_o) == 0
    assert np.array_equal(np.fromfile(d / "arena.out", dtype=np.uint8), arena_o)
    assert np.array_equal(np.fromfile(d / "fresh.out", dtype=np.uint8), fresh_o)


@pytest.mark.gpu
def test_python_usage_example_runs():
    """The usage example (tests/example_usage.py, also printed in the README)
    runs as written: a Kimi-Linear layout, one request's two chunks stored
    into objects and loaded into other blocks, a page checked."""
    import example_usage
    out = example_usage.run("cuda")
    assert out == {"C": 944, "num_blocks": 64, "status": 0}
