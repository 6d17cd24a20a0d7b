"""The C-ABI library builds, loads and exports every function include/pdattn.h
declares; host-side argument checks reject bad calls before any launch.

CPU only: nothing here launches a kernel.
"""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pdattn.h")


@pytest.fixture(scope="module")
def lib():
    from paged_gqa_decode_step_gb300 import build
    path = build.build()
    from paged_gqa_decode_step_gb300 import binding
    assert os.path.samefile(binding.LIB_PATH, path)
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pdattn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pdattn_rope_write_kv", "pdattn_decode", "pdattn_decode_fused", "pdattn_workspace_size",
                     "pdattn_check_status", "pdattn_last_error", "pdattn_rope_tables", "pdattn_plan",
                     "pdattn_attend"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r" T (pdattn_\w+)", out.stdout))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib.lib, name) is not None


def test_header_compiles_as_c():
    src = '#include "pdattn.h"\nint main(void) { pdattn_params p; (void)p; return (int)PDATTN_OK; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-x", "c", "-", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include")], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_params_struct_layout_matches_header(lib):
    # offsets of the C struct, computed by the C compiler
    src = r'''
#include <stddef.h>
#include <stdio.h>
#include "pdattn.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(pdattn_params), offsetof(pdattn_params, scale),
         offsetof(pdattn_params, rope_cos), offsetof(pdattn_params, rope_sin),
         offsetof(pdattn_params, rope_len), offsetof(pdattn_params, chunk_pages),
         offsetof(pdattn_params, sinks));
  return 0;
}
'''
    exe = os.path.join(ROOT, "paged_gqa_decode_step_gb300", "_build", "layout_probe")
    r = subprocess.run(["gcc", "-x", "c", "-", "-o", exe, "-I", os.path.join(ROOT, "include")],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True).stdout.split()]
    P = lib.Params
    want = [ctypes.sizeof(P), P.scale.offset, P.rope_cos.offset, P.rope_sin.offset, P.rope_len.offset,
            P.chunk_pages.offset, P.sinks.offset]
    assert got == want


def _p(lib, **kw):
    import torch
    base = dict(rows=2, heads=8, kv_heads=2, head_dim=64, pages_per_row=4, num_pages=8, dtype=torch.bfloat16)
    base.update(kw)
    return lib.make_params(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(heads=6, kv_heads=4), 1),          # heads % kv_heads != 0
    (dict(head_dim=0), 1),
    (dict(head_dim=96), 2),                 # unsupported head dim
    (dict(heads=32, kv_heads=2), 2),        # group of 16 > 8
    (dict(num_pages=0), 1),
    (dict(chunk_pages=65), 1),
    (dict(rows=-1), 1),
])
def test_host_validation_rejects_before_launch(lib, kw, status):
    p = _p(lib, **kw)
    null = ctypes.c_void_p(0)
    rc = lib.lib.pdattn_decode_fused(ctypes.byref(p), *([null] * 9), 0, null)
    assert rc == status
    assert lib.lib.pdattn_last_error()
    assert lib.lib.pdattn_workspace_size(ctypes.byref(p)) == 0


def test_null_pointers_rejected(lib):
    p = _p(lib)
    null = ctypes.c_void_p(0)
    assert lib.lib.pdattn_decode_fused(ctypes.byref(p), *([null] * 9), 0, null) == 1
    assert b"NULL" in lib.lib.pdattn_last_error()
    assert lib.lib.pdattn_rope_tables(-1.0, 64, 8, 0, null, null, null) == 1
    assert lib.lib.pdattn_check_status(null, null) == 1


def test_zero_rows_is_a_no_op(lib):
    p = _p(lib, rows=0)
    null = ctypes.c_void_p(0)
    assert lib.lib.pdattn_decode_fused(ctypes.byref(p), *([null] * 9), 0, null) == 0
    assert lib.lib.pdattn_last_launch_count() == 0


def test_workspace_layout_bound_covers_every_plan():
    # The planner's item count never exceeds the workspace bound: replay its
    # chunking rule on random position sets (host arithmetic only).
    import math
    import random
    rnd = random.Random(3)
    items_per_cta, chunk_max = 4, 64
    for _ in range(300):
        R, Hk, Pg, grid = rnd.randint(1, 300), rnd.choice([1, 2, 8, 12]), rnd.randint(1, 128), rnd.choice([1, 20, 152])
        pos = [rnd.randint(0, Pg * 64 - 1) for _ in range(R)]
        W = window = 0
        window = rnd.choice([0, 0, 1, 100, 1000])
        n = []
        for p in pos:
            lo = max(0, p - window + 1) if window > 0 else 0
            n.append(p // 64 - lo // 64 + 1)
        W = sum(n) * Hk
        few_pairs = R * Hk < 2 * grid
        if not few_pairs and max(n) * grid <= 2 * W:
            C = chunk_max                  # rows kept whole
        else:
            per = (2 * items_per_cta if few_pairs else items_per_cta) * grid
            C = min(max(math.ceil(W / per), 1), chunk_max)
        items = sum(Hk * math.ceil(x / C) for x in n)
        # at most one empty first-wave item per CTA (a row with a bad position)
        items += min(grid, R * Hk) if R <= 512 else 0
        bound = max(2 * items_per_cta * grid + R * Hk, R * Hk * math.ceil(Pg / chunk_max)) + grid
        assert items <= bound


def test_prefill_host_validation(lib):
    import torch
    null = ctypes.c_void_p(0)
    f = lib.lib.pdattn_prefill_paged
    p = _p(lib, dtype=torch.float32)
    assert f(ctypes.byref(p), 4, *([null] * 11), 0, null) == 2        # tensor-core path: bf16 only
    p = _p(lib)
    assert f(ctypes.byref(p), -1, *([null] * 11), 0, null) == 1
    assert f(ctypes.byref(p), 0, *([null] * 11), 0, null) == 0         # no tokens: nothing launched
    assert lib.lib.pdattn_last_launch_count() == 0
    assert f(ctypes.byref(p), 4, *([null] * 11), 0, null) == 1
    assert b"NULL" in lib.lib.pdattn_last_error()
    # workspace: control block, two tile lists and the rotated queries
    n = lib.lib.pdattn_prefill_workspace_size(ctypes.byref(p), 1000)
    assert n >= 256 + 2 * 32 * 1000 + 2 * 1000 * 8 * 64 and n % 256 == 0
    assert lib.lib.pdattn_prefill_workspace_size(ctypes.byref(p), -1) == 0


def test_packed_host_validation(lib):
    import torch
    null = ctypes.c_void_p(0)
    f = lib.lib.pdattn_packed
    p = _p(lib, dtype=torch.float32)
    assert f(ctypes.byref(p), 4, *([null] * 7), 0, null) == 2         # tensor-core path: bf16 only
    p = _p(lib, pages_per_row=0, num_pages=0)                           # cache fields are not read
    assert f(ctypes.byref(p), -1, *([null] * 7), 0, null) == 1
    assert f(ctypes.byref(p), 0, *([null] * 7), 0, null) == 0
    assert lib.lib.pdattn_last_launch_count() == 0
    assert f(ctypes.byref(p), 4, *([null] * 7), 0, null) == 1
    assert b"NULL" in lib.lib.pdattn_last_error()
    n = lib.lib.pdattn_packed_workspace_size(ctypes.byref(p), 1000)
    # control, two tile lists, rotated q and k, padded ids and positions, block summaries
    assert n >= 256 + 2 * 32 * 1000 + 2 * 1000 * (8 + 2) * 64 + 2 * 4 * 1024 + 16 * 16 and n % 256 == 0


def test_layer_struct_layout_matches_header(lib):
    src = r"""
#include <stddef.h>
#include <stdio.h>
#include "pdattn.h"
int main(void) {
  printf("%zu %zu %zu %zu %d\n", sizeof(pdattn_layer), offsetof(pdattn_layer, out),
         offsetof(pdattn_layer, window), offsetof(pdattn_layer, sinks), PDATTN_LAYERS_PER_LAUNCH);
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "l.c")
        exe = os.path.join(d, "l")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    L = lib.Layer
    assert got == [ctypes.sizeof(L), L.out.offset, L.window.offset, L.sinks.offset, lib.LAYERS_PER_LAUNCH]


def test_decode_layers_host_validation(lib):
    p = lib.make_params(4, 32, 8, 128, 8, 40, torch.bfloat16)
    null = ctypes.c_void_p(0)
    f = lib.lib.pdattn_decode_layers
    # zero layers: a no-op; NULL layer array or pointers: rejected before any launch
    assert f(ctypes.byref(p), 0, None, null, null, null, 0, null) == lib.OK
    assert lib.last_launch_count() == 0
    assert f(ctypes.byref(p), 2, None, null, null, null, 0, null) == lib.EINVAL
    arr = (lib.Layer * 2)()
    assert f(ctypes.byref(p), 2, arr, ctypes.c_void_p(256), ctypes.c_void_p(256), null, 0, null) == lib.EINVAL
    assert b"layer 0" in lib.lib.pdattn_last_error()
    assert f(ctypes.byref(p), -1, arr, null, null, null, 0, null) == lib.EINVAL
    assert lib.last_launch_count() == 0
    assert lib.lib.pdattn_layers_workspace_size(ctypes.byref(p), -1) == 0
    if torch.cuda.is_available():
        # the workspace covers up to one launch's layers
        n1 = lib.lib.pdattn_layers_workspace_size(ctypes.byref(p), 1)
        n32 = lib.lib.pdattn_layers_workspace_size(ctypes.byref(p), 32)
        n64 = lib.lib.pdattn_layers_workspace_size(ctypes.byref(p), 64)
        assert 0 < n1 < n32 == n64
