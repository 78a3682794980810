"""The C-ABI library builds, loads and exports every entry point its headers
declare; host-side validation and planning behave as documented.  No GPU."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"^(?:hd_status|const char \*)\s*(\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("hybrid_decode_init", "rope_append_kv", "decode_attn_sliding", "decode_attn_full",
                 "decode_step", "hybrid_decode_destroy", "hd_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    nm = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True,
                        check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", nm, re.M))
    for name in declared_functions():
        assert name in exported, f"{name} is declared but not exported"
        assert hasattr(lib, name)


def test_status_strings(hd):
    assert hd.hd_status_string(0) == "ok"
    assert hd.hd_status_string(3) == "capacity exceeded"


def _cfg(hd, **kw):
    base = dict(layer_types=[hd.HD_SLIDING] * 3 + [hd.HD_FULL], max_batch=4, max_context=4096)
    base.update(kw)
    return hd.Config(**base)


def test_validate_config_mirrors_post_init(hd):
    assert hd.hd_validate_config(_cfg(hd)) == 0
    assert hd.hd_validate_config(_cfg(hd, num_q_heads=6, num_kv_heads=4)) == 1   # not a multiple
    assert hd.hd_validate_config(_cfg(hd, layer_types=[0, 1, 7])) == 1          # unknown layer type
    assert hd.hd_validate_config(_cfg(hd, cache_layout=3)) == 1                 # unknown layout
    assert hd.hd_validate_config(_cfg(hd, rotary_dim_full=63)) == 1             # odd rotary dim
    assert hd.hd_validate_config(_cfg(hd, rotary_dim_sliding=512)) == 1         # beyond head_dim
    assert hd.hd_validate_config(_cfg(hd, rope_theta_full=0.0)) == 1
    assert hd.hd_validate_config(_cfg(hd, max_batch=0)) == 1
    assert hd.hd_validate_config(_cfg(hd, head_dim=128, rotary_dim_sliding=128)) == 2
    assert hd.hd_validate_config(_cfg(hd, num_q_heads=32, num_kv_heads=2)) == 2  # group 16
    for g in (1, 2, 4, 8):
        assert hd.hd_validate_config(_cfg(hd, num_q_heads=2 * g, num_kv_heads=2)) == 0


@pytest.mark.parametrize("batch,max_keys", [(1, 4097), (64, 32769), (4, 131073), (256, 8193),
                                            (64, 511), (1, 1), (2, 0), (256, 512)])
def test_plan_split_covers_the_keys(hd, batch, max_keys):
    ck, nc = hd.hd_plan_split(batch, 2, max_keys, 152)
    assert ck in (64, 128, 256, 512, 1024, 2048)
    assert nc * ck >= max_keys and (nc - 1) * ck < max(max_keys, 1)


def test_plan_split_long_context_uses_many_chunks(hd):
    ck, nc = hd.hd_plan_split(4, 2, 131073, 152)
    assert nc >= 64


def test_plan_split_shapes(hd):
    assert hd.hd_plan_split(4, 2, 131073, 152) == (2048, 65)   # long context: >= 64 chunks
    assert hd.hd_plan_split(64, 2, 32769, 152) == (2048, 17)   # batch-64 full layers
    assert hd.hd_plan_split(64, 2, 511, 152) == (512, 1)       # batch-64 ring layers: one chunk
    assert hd.hd_plan_split(1, 2, 4097, 152) == (64, 65)       # batch 1: many short chunks


def _spark_keys(full_keys, sliding_keys=511):
    return [sliding_keys, sliding_keys, sliding_keys, full_keys] * 7


def test_step_plan_shapes(hd):
    """The step grid's chunk plan on the benchmark shapes (152 SMs)."""
    # batch 64, contexts up to 32768: the longest bf16 chunk (sliding layers one chunk)
    assert hd.hd_plan_step_split(_spark_keys(32768), 64, 2, 4, 152) == 2048
    # E4M3: the same bytes per chunk, twice the keys
    assert hd.hd_plan_step_split(_spark_keys(32768), 64, 2, 4, 152, kv_dtype=hd.HD_KV_FP8_E4M3) == 4096
    # batch 1 at 4096: 140 CTAs of up to 640 keys, one wave on 152 SMs
    assert hd.hd_plan_step_split(_spark_keys(4096), 1, 2, 4, 152) == 640
    # 7 full layers at 131072, batch 4: 2048-key chunks (64 per sequence)
    assert hd.hd_plan_step_split([131072] * 7, 4, 2, 4, 152) == 2048


@pytest.mark.parametrize("batch,full_keys", [(1, 1), (1, 700), (2, 4096), (3, 20000), (64, 32768), (256, 8192)])
def test_step_plan_is_a_multiple_of_64_within_the_limit(hd, batch, full_keys):
    for kv, cmax in ((hd.HD_KV_BF16, 2048), (hd.HD_KV_FP8_E4M3, 4096)):
        c = hd.hd_plan_step_split(_spark_keys(full_keys), batch, 2, 4, 152, kv_dtype=kv)
        assert c % 64 == 0 and 64 <= c <= cmax


def test_step_plan_rolled_windows_take_one_chunk(hd):
    """Rolled windows read their 511 keys in one chunk whatever the plan's size:
    the plan may pick chunks shorter than 511 for the other layers."""
    keys = _spark_keys(4096)
    one = [k == 511 for k in keys]
    c = hd.hd_plan_step_split(keys, 1, 2, 4, 152, one_chunk=one)
    assert c % 64 == 0
    assert max(c, 511) >= 511


def test_step_plan_rejects_bad_arguments(hd):
    with pytest.raises(Exception):
        hd.hd_plan_step_split([], 1, 2, 4, 152)
    with pytest.raises(Exception):
        hd.hd_plan_step_split([100], 0, 2, 4, 152)
    with pytest.raises(Exception):
        hd.hd_plan_step_split([100], 1, 2, 33, 152)   # more rows than a pass takes
    with pytest.raises(Exception):
        hd.hd_plan_step_split([-1], 1, 2, 4, 152)


def test_binding_structs_match_the_header(hd, tmp_path):
    """Every struct field of the ctypes binding sits at the offset the C compiler
    gives it from include/hybrid_decode.h, and the struct sizes agree."""
    structs = {"hd_config": hd.hd_config, "hd_kv_cache": hd.hd_kv_cache, "hd_layer_io": hd.hd_layer_io}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "hybrid_decode.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        s, f, v = line.split()
        got[(s, f)] = int(v)
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert got[(name, field)] == getattr(cls, field).offset, (name, field)


def test_config_rejects_an_unknown_kv_dtype(hd):
    cfg = hd.Config(layer_types=[0, 1], kv_dtype=hd.HD_KV_FP8_E4M3)
    assert hd.hd_validate_config(cfg) == 0
    cfg.kv_dtype = 2
    assert hd.hd_validate_config(cfg) == 1


def test_static_scratch_plan_counts_the_scratch_it_needs(hd):
    """The allocation-free entry point's scratch: one (o[256], m, l) partial per
    (sequence, query head, chunk), one ticket per (sequence, kv head) and the
    error word, against the array's size; every key is covered by the chunks."""
    for B, Hq, Hkv, mc in [(1, 8, 2, 0), (6, 8, 2, 9000), (64, 16, 2, 4096), (256, 8, 2, 8191), (3, 2, 2, 2048)]:
        nbytes, chunk, chunks, st = hd.decode_attn_full_static_scratch_plan(B, Hq, Hkv, mc, 152)
        assert st == 0, (B, Hq, Hkv, mc)
        assert chunk * chunks >= mc + 1 and chunk * (chunks - 1) < mc + 1
        assert nbytes == B * Hq * chunks * (256 * 4 + 8) + B * Hkv * 4 + 4
        assert nbytes <= hd.HD_STATIC_SCRATCH_BYTES


def test_static_scratch_plan_refuses_beyond_the_array(hd):
    # 16 sequences, group 8, 131072 keys: 64 chunks of 2048 keys per sequence
    nbytes, chunk, chunks, st = hd.decode_attn_full_static_scratch_plan(16, 64, 8, 131071, 152)
    assert (st, chunk, chunks) == (3, 2048, 64)
    assert nbytes == 16 * 64 * 64 * 1032 + 16 * 8 * 4 + 4 > hd.HD_STATIC_SCRATCH_BYTES
    # the largest context that still fits at this shape, found by bisection, and the next one refused
    lo, hi = 0, 131071
    while lo + 1 < hi:
        mid = (lo + hi) // 2
        if hd.decode_attn_full_static_scratch_plan(16, 64, 8, mid, 152)[3] == 0:
            lo = mid
        else:
            hi = mid
    assert hd.decode_attn_full_static_scratch_plan(16, 64, 8, lo, 152)[0] <= hd.HD_STATIC_SCRATCH_BYTES
    nb, _, _, st = hd.decode_attn_full_static_scratch_plan(16, 64, 8, hi, 152)
    assert st == 3 and nb > hd.HD_STATIC_SCRATCH_BYTES


def test_static_scratch_plan_rejects_bad_shapes(hd):
    plan = hd.decode_attn_full_static_scratch_plan
    assert plan(0, 8, 2, 10, 152)[3] == 1          # no sequences
    assert plan(4, 6, 4, 10, 152)[3] == 1          # heads not a multiple
    assert plan(4, 8, 2, -1, 152)[3] == 1          # negative context bound
    assert plan(4, 8, 2, 10, 0)[3] == 1            # no SMs
    assert plan(4, 32, 2, 10, 152)[3] == 2         # group 16


@pytest.mark.parametrize("rows", [16, 32])
def test_step_plan_multi_token_passes_fit_their_ring(hd, rows):
    """Multi-token passes of 16 rows (six-stage ring) and 32 rows (the tcgen05 pass's
    160 KiB ring): the step plan picks a chunk whose combine fits that ring, for the
    benchmark's batch-64 step and the 131k-context case."""
    for keys, batch in ((_spark_keys(32768 + 8), 64), ([131072 + 8] * 7, 4)):
        c = hd.hd_plan_step_split(keys, batch, 2, rows, 152, multi_token=True)
        assert c % 64 == 0 and 64 <= c <= 2048
