"""The bulk-copy (TMA) engine, a build-time alternative to the default
vector engine (LMC_ENGINE=1): cp.async.bulk global->shared->global through
an mbarrier-tracked ring of shared-memory stages. It is compiled into a
separate library in a temporary directory, bound for the duration of these
tests only, and checked byte for byte against the CPU oracle."""
import importlib.util
import os

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


ENGINES = {
    "bulk": ["-DLMC_ENGINE=1", "-DLMC_TILE_BYTES=32768", "-DLMC_BULK_STAGES=4", "-DLMC_BULK_CTAS_PER_SM=1"],
}


@pytest.fixture(scope="module", params=sorted(ENGINES))
def bulk_lmc(request, tmp_path_factory, lmc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    spec = importlib.util.spec_from_file_location("lmc_build", os.path.join(ROOT, "state_cache_paging_gb300",
                                                                             "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    so = str(tmp_path_factory.mktemp(request.param) / f"liblmc_{request.param}.so")
    b.build_library(extra_nvcc=ENGINES[request.param], out_path=so)
    lmc._use_library(so)
    try:
        yield lmc
    finally:
        torch.cuda.synchronize()
        lmc._use_library(lmc.LIB_PATH)


def test_bulk_engine_tiny_workload_exact(bulk_lmc):
    import test_gpu_parity as T
    inp, Lp = T.case_inputs(W.CONFIGS[0])
    T._full_exact(bulk_lmc, inp, Lp)


@pytest.mark.parametrize("t", range(6))
def test_bulk_engine_random_specs_exact(bulk_lmc, t):
    import test_gpu_parity as T
    rng = np.random.default_rng(5000 + t)
    cfg = T._random_cfg(rng, t)
    inp, Lp = T.case_inputs(cfg, split=bool(t % 2))
    T._full_exact(bulk_lmc, inp, Lp)


def test_bulk_engine_error_paths(bulk_lmc):
    import test_gpu_parity as T
    T.test_error_paths_match_oracle(bulk_lmc)


def test_bulk_engine_large_pages_exact(bulk_lmc):
    import test_gpu_parity as T
    T.test_large_pages_exact(bulk_lmc)


def test_bulk_engine_odd_sizes_and_copies_exact(bulk_lmc):
    """Tiles that are only 16-byte aligned (odd page sizes) and in-pool block
    copies through the alternative engine."""
    import test_gpu_parity as T
    T.test_odd_page_sizes_exact(bulk_lmc)
    T.test_copy_blocks_exact(bulk_lmc, 7)


@pytest.mark.parametrize("packed", [False, True])
def test_bulk_engine_16_byte_pages_exact(bulk_lmc, packed):
    """Pages that are 16-byte but not 32-byte multiples (MLA 3 x 48 B, KDA
    16 + 4096 B): vector tiles that cannot take 32-byte accesses."""
    import test_gpu_parity as T
    kda = {"kind": "KDA", "token_bytes": 0, "conv_bytes": 16, "rec_bytes": 4096, "window": 0}
    spec = [kda, kda, W.mla(48), kda, W.mla(48)]
    cfg = W.Config(240 + int(packed), "16B", spec, N=3, requested_chunk=6, packed=packed, num_requests=3,
                   lengths="fixed", fixed_lengths=(40, 61, 25), seed=41)
    inp, Lp = T.case_inputs(cfg)
    T._full_exact(bulk_lmc, inp, Lp)
