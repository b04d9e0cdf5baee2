"""Each plausible mistake planted in a copy of the CPU oracle must make at
least one pin fail. The mutants are compiled from a copy in a temporary
directory and run in a child process, so a mutant that crashes counts as
caught and cannot take the test run down."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oracle.c")

MUTANTS = [
    ("negotiation does not round up", "k += 1;", "k += 0;"),
    ("non-positive request negotiates to 0", "*out = N;\n        return OR_OK;", "*out = 0;\n        return OR_OK;"),
    ("budget boundary 2N included", "if (max_batched < 2 * N)", "if (max_batched <= 2 * N)"),
    ("paged page one token short", "return N * l->token_bytes;", "return (N - 1) * l->token_bytes;"),
    ("KDA page drops conv_state", "return l->conv_bytes + l->rec_bytes;", "return l->rec_bytes;"),
    ("padded page is the first layer's", "if (L->real_bytes[i] > page)", "if (i == 0)"),
    ("padded slab base ignores num_blocks", "L->base[i] = (int64_t)L->slot[i] * page * nb;",
     "L->base[i] = (int64_t)L->slot[i] * page;"),
    ("runs per spec rounded down", "runs = (cnt + smallest - 1) / smallest;", "runs = cnt / smallest + (cnt % smallest > 1);"),
    ("sliding windows merged", "return a->window == b->window;", "return 1;"),
    ("packed offset counted after the page", "offset_in_group[i] = group_total[k];\n                        group_total[k] += L->real_bytes[i];",
     "group_total[k] += L->real_bytes[i];\n                        offset_in_group[i] = group_total[k] - L->real_bytes[0];"),
    ("packed stride is the first group's", "if (group_total[k] > stride)", "if (k == 0)"),
    ("KDA snapshot from the object's first block", "int64_t pos = first + nb - 1;", "int64_t pos = first;"),
    ("paged blocks reversed in the object", "int64_t pos = first + j;", "int64_t pos = first + (nb - 1 - j);"),
    ("every-block snapshots all from the last block", "int64_t pos = first + s;", "int64_t pos = first + nb - 1;"),
    ("block jobs start at chunk * nb", "int64_t first = sh->first_is_block ? c : c * nb;", "int64_t first = c * nb;"),
    ("copy writes the source", "memmove(pool + L->base[i] + dst * L->stride[i],\n                        pool + L->base[i] + src * L->stride[i]",
     "memmove(pool + L->base[i] + src * L->stride[i],\n                        pool + L->base[i] + dst * L->stride[i]"),
    ("copy skips a group's last layer", "                if (L->kv_group[i] != g)\n                    continue;\n                memmove",
     "                if (L->kv_group[i] != g || i == L->num_layers - 1)\n                    continue;\n                memmove"),
    ("codec rounds half away from zero", "q = rintf(v / scale);", "q = roundf(v / scale);"),
    ("codec scales by 128", "float scale = amax / 127.0f;", "float scale = amax / 128.0f;"),
    ("codec does not clamp", "                if (q > 127.0f)\n                    q = 127.0f;", "                if (0)\n                    q = 127.0f;"),
    ("codec drops the conv window", "    memcpy(rec, page, (size_t)l->conv_bytes);", "    memset(rec, 0, (size_t)l->conv_bytes);"),
    ("codec record has no scales", "    return l->conv_bytes + 4 * rows + rows * d;", "    return l->conv_bytes + rows * d;"),
    ("decoder ignores the scale", "float v = (float)codes[r * d + j] * scale;", "float v = (float)codes[r * d + j];"),
    ("padded attention always allowed", "L->page_bytes[i] > L->real_bytes[i] && !attn_indexes_by_stride",
     "L->page_bytes[i] > L->real_bytes[i] && !attn_indexes_by_stride && 0"),
    ("packed state pages always allowed", "if (!attention && !state_pages_strided_ok)", "if (0)"),
    ("copy accepts block ids past the pool", "dst < 0 || dst >= L->num_blocks", "dst < 0 || dst > L->num_blocks + 1000000"),
    ("page copy one byte short", "memcpy(obj_bytes, page, (size_t)L->real_bytes[layer]);",
     "memcpy(obj_bytes, page, (size_t)L->real_bytes[layer] - 1);"),
    ("misaligned object offsets accepted", "job->offset % 16 != 0 ||", ""),
    ("block id upper bound off by one", "block >= L->num_blocks", "block > L->num_blocks"),
    ("object size counts KDA per block", "        if (L->layers[i].kind == OR_KDA && !kda_every)\n            total += page;",
     "        if (0)\n            total += page;"),
    ("every-block snapshots stored raw under the codec",
     "else if (sh->q8_row > 0)\n                            *status |= q8_page(",
     "else if (0)\n                            *status |= q8_page("),
    ("every-block INT8 records advance by the raw page",
     "cursor += sh->q8_row > 0 ? q8_record_bytes(&L->layers[i], sh->q8_row)\n                                                 : L->real_bytes[i];",
     "cursor += L->real_bytes[i];"),
    ("copies may write a block another pair reads",
     "p->dst_block == o->dst_block || p->dst_block == o->src_block", "p->dst_block == o->dst_block"),
    ("copies may write one block twice",
     "p->dst_block == o->dst_block || p->dst_block == o->src_block", "p->dst_block == o->src_block"),
    ("copy collisions looked for only inside a KV group", "if ((h == g && t == q) ||", "if (h != g || t == q ||"),
    ("disjoint check marks a KDA layer's first position", "lo = hi - 1;", "lo = lo + 0;"),
    ("disjoint check drops a chunk's last paged position", "pos < hi && pos < T->num_cols[k]",
     "pos < hi - 1 + (L->layers[i].kind == OR_KDA) && pos < T->num_cols[k]"),
    ("block-form disjoint check ignores every-block snapshots",
     "if (L->layers[i].kind == OR_KDA && !sh->kda_every)\n                    lo = hi - 1;",
     "if (L->layers[i].kind == OR_KDA)\n                    lo = hi - 1;"),
]


@pytest.mark.parametrize("what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, what, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new, 1))
    so = str(tmp_path / "libmutant.so")
    oracle.build(out_path=so, src_path=str(mutated))
    r = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), so],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant survived every pin: {what}"
