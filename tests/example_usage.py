"""The Python usage example shown in the README, as a module the tests run.

A Kimi-Linear layout (18 KDA + 6 MLA layers, N = 944, padded, 64 blocks),
one request's two chunks stored into per-object-group objects and loaded
into other blocks of a second pool, one page compared. run() returns the
values a test checks.
"""


def run(device="cuda"):
    import numpy as np
    import torch

    import state_cache_paging_gb300 as lmc

    kda = {"kind": "KDA", "conv_bytes": 12288 * 3 * 2, "rec_bytes": 32 * 128 * 128 * 4}
    mla = {"kind": "MLA", "token_bytes": (512 + 64) * 2}
    layers = [kda, kda, kda, mla] * 6                          # model order (Kimi-Linear)
    N = 944
    C = lmc.lmc_negotiate_chunk(944, N)                         # smallest multiple of N >= request
    L = lmc.lmc_layout_build(layers, N, packed=False, mem_bytes=64 * 6 * 2170880)   # 64 blocks
    pool = torch.randint(0, 256, (L.pool_bytes,), dtype=torch.uint8, device=device)

    # one request holding two chunks: per KV group an int32 block table [requests, positions]
    # (groups share pages at equal block ids, so each group gets its own blocks)
    tables = [torch.tensor([[2 * k, 2 * k + 1]], dtype=torch.int32, device=device)
              for k in range(L.num_kv_groups)]
    # per object group one 16-byte job (request, chunk, arena offset) per object
    sizes = [L.object_bytes(C, g) for g in range(L.num_object_groups)]
    jobs_np, off = [np.zeros(2, dtype=lmc.JOB_DTYPE) for _ in sizes], 0
    for g, J in enumerate(jobs_np):
        for c in range(2):
            J[c] = (0, c, off)
            off += sizes[g]
    jobs = [lmc.jobs_to_device(J, device) for J in jobs_np]
    arena = torch.empty(off, dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)

    lmc.lmc_store(L, C, pool, tables, jobs, arena, status)          # gather into objects
    fresh, new_tables = torch.zeros_like(pool), [t + 16 for t in tables]
    lmc.lmc_load(L, C, fresh, new_tables, jobs, arena, status)      # scatter into other blocks
    torch.cuda.synchronize()
    assert status.item() == 0
    i = 3                                                            # the first MLA layer, chunk 1
    src = L.base[i] + int(tables[L.kv_group[i]][0, 1]) * L.stride[i]
    dst = L.base[i] + int(new_tables[L.kv_group[i]][0, 1]) * L.stride[i]
    assert torch.equal(pool[src:src + L.real_bytes[i]], fresh[dst:dst + L.real_bytes[i]])
    return {"C": C, "num_blocks": L.num_blocks, "status": int(status.item())}
