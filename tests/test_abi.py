"""The C-ABI library loads and exports what include/ssattn.h declares (CPU).

No compute call reaches a GPU here: only host-side logic (argument
validation that rejects before any device work, the factor fit, lambda,
status strings)."""
import ctypes
import math
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssattn.h")


@pytest.fixture(scope="module")
def capi():
    import block_sparse_attention_sm_gb300 as ss
    from block_sparse_attention_sm_gb300 import capi

    ss.build()
    capi.load()
    return capi


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(capi):
    decl = declared_functions()
    assert len(decl) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\S+)$", out, flags=re.M))
    missing = [f for f in decl if f not in exported]
    assert not missing, f"declared but not exported: {missing}"
    assert set(capi.EXPORTS) == set(decl)
    for f in decl:
        assert hasattr(capi.load(), f)


def test_status_strings(capi):
    for st in range(6):
        assert capi.ss_status_string(st)
    assert "invalid" in capi.ss_status_string(capi.SS_ERR_INVALID_ARG)


def test_lambda_and_fit(capi):
    # §The threshold: threshold = factor / seqlen, factor = A exp(B s)
    assert math.isclose(capi.ss_lambda(2.0, 1.5, 0.7, 4096), 2.0 * math.exp(1.05) / 4096,
                        rel_tol=1e-6)
    s = [0.5, 0.7, 0.9]
    a = [3.0 * math.exp(2.0 * x) for x in s]
    st, A, B = capi.ss_fit_factor(s, a)
    assert st == capi.SS_OK
    assert math.isclose(A, 3.0, rel_tol=1e-5) and math.isclose(B, 2.0, rel_tol=1e-5)
    assert capi.ss_fit_factor([0.5], [1.0])[0] == capi.SS_ERR_INVALID_ARG
    assert capi.ss_fit_factor([0.5, 0.6], [1.0, -1.0])[0] == capi.SS_ERR_INVALID_ARG


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced here


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), "SS_ERR_INVALID_ARG"),
    (dict(q=FAKE + 8), "SS_ERR_INVALID_ARG"),          # misaligned
    (dict(Lq=0), "SS_ERR_INVALID_ARG"),                # empty input
    (dict(B=0), "SS_ERR_INVALID_ARG"),
    (dict(Hq=3, Hkv=2), "SS_ERR_INVALID_ARG"),         # Hq % Hkv != 0
    (dict(lam=1.5), "SS_ERR_INVALID_ARG"),
    (dict(lam=float("nan")), "SS_ERR_INVALID_ARG"),
    (dict(lam=-0.1), "SS_ERR_INVALID_ARG"),
    (dict(scale=0.0), "SS_ERR_INVALID_ARG"),
    (dict(d=96), "SS_ERR_UNSUPPORTED"),
])
def test_prefill_rejects_before_launch(capi, kw, expect):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, Hq=2, Hkv=1, Lq=128, Lk=128, d=128,
                scale=0.1, causal=0, lam=0.01)
    args.update(kw)
    st = capi.ss_attn_prefill(args["q"], args["k"], args["v"], args["o"], args["B"], args["Hq"],
                              args["Hkv"], args["Lq"], args["Lk"], args["d"], args["scale"],
                              args["causal"], args["lam"], None, 0)
    assert st == getattr(capi, expect)


@pytest.mark.parametrize("kw,expect", [
    (dict(S=0), "SS_ERR_INVALID_ARG"),
    (dict(Lk=0), "SS_ERR_INVALID_ARG"),
    (dict(Hq=258, Hkv=2), "SS_ERR_UNSUPPORTED"),      # vote group > 128 (MMA rows)
    (dict(Hq=66, Hkv=2, d=64), "SS_ERR_UNSUPPORTED"),  # vote group > 32 at d = 64
    (dict(S=4, ws=None), "SS_ERR_WORKSPACE"),
    (dict(S=4, ws_bytes=16), "SS_ERR_WORKSPACE"),
])
def test_decode_rejects_before_launch(capi, kw, expect):
    args = dict(B=2, Hq=8, Hkv=2, Lk=1000, d=128, S=1, ws=FAKE, ws_bytes=1 << 30)
    args.update(kw)
    st = capi.ss_attn_decode(FAKE, FAKE, FAKE, FAKE, args["B"], args["Hq"], args["Hkv"],
                             args["Lk"], args["d"], 0.1, 0.01, args["S"], None, args["ws"],
                             args["ws_bytes"], 0)
    assert st == getattr(capi, expect)


@pytest.mark.parametrize("kw,expect", [
    (dict(table=None), "SS_ERR_INVALID_ARG"),
    (dict(lens=None), "SS_ERR_INVALID_ARG"),
    (dict(num_pages=0), "SS_ERR_INVALID_ARG"),
    (dict(max_pages=0), "SS_ERR_INVALID_ARG"),
    (dict(a=-1.0), "SS_ERR_INVALID_ARG"),
    (dict(a=float("inf")), "SS_ERR_INVALID_ARG"),
    (dict(k=FAKE + 4), "SS_ERR_INVALID_ARG"),
    (dict(d=96), "SS_ERR_UNSUPPORTED"),
    (dict(Hq=258, Hkv=2), "SS_ERR_UNSUPPORTED"),
    (dict(Hq=66, Hkv=2, d=64), "SS_ERR_UNSUPPORTED"),
    (dict(S=4, ws=None), "SS_ERR_WORKSPACE"),
])
def test_paged_decode_rejects_before_launch(capi, kw, expect):
    args = dict(k=FAKE, table=FAKE, lens=FAKE, B=2, Hq=8, Hkv=2, num_pages=10, max_pages=4, d=128,
                a=1.0, S=1, ws=FAKE, ws_bytes=1 << 30)
    args.update(kw)
    st = capi.ss_attn_decode_paged(FAKE, args["k"], FAKE, args["table"], args["lens"], FAKE,
                                   args["B"], args["Hq"], args["Hkv"], args["num_pages"],
                                   args["max_pages"], args["d"], 0.1, args["a"], args["S"], None,
                                   args["ws"], args["ws_bytes"], stream=0)
    assert st == getattr(capi, expect)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), "SS_ERR_INVALID_ARG"),
    (dict(kv=FAKE + 8), "SS_ERR_INVALID_ARG"),     # misaligned cache
    (dict(B=0), "SS_ERR_INVALID_ARG"),
    (dict(Lk=0), "SS_ERR_INVALID_ARG"),
    (dict(S=0), "SS_ERR_INVALID_ARG"),
    (dict(lam=1.5), "SS_ERR_INVALID_ARG"),
    (dict(scale=0.0), "SS_ERR_INVALID_ARG"),
    (dict(Hq=65), "SS_ERR_UNSUPPORTED"),            # more heads than one staged query block
    (dict(d_latent=256), "SS_ERR_UNSUPPORTED"),
    (dict(d_rope=32), "SS_ERR_UNSUPPORTED"),
    (dict(S=4, ws_bytes=16), "SS_ERR_WORKSPACE"),
])
def test_mla_decode_rejects_before_launch(capi, kw, expect):
    args = dict(q=FAKE, kv=FAKE, B=2, Hq=16, Lk=1000, d_latent=512, d_rope=64, scale=0.07,
                lam=0.01, S=1, ws=FAKE, ws_bytes=1 << 30)
    args.update(kw)
    st = capi.ss_attn_mla_decode(args["q"], args["kv"], FAKE, args["B"], args["Hq"], args["Lk"],
                                 args["d_latent"], args["d_rope"], args["scale"], args["lam"],
                                 args["S"], None, args["ws"], args["ws_bytes"], stream=0)
    assert st == getattr(capi, expect)


@pytest.mark.parametrize("kw,expect", [
    (dict(table=None), "SS_ERR_INVALID_ARG"),
    (dict(lens=None), "SS_ERR_INVALID_ARG"),
    (dict(num_pages=0), "SS_ERR_INVALID_ARG"),
    (dict(max_pages=0), "SS_ERR_INVALID_ARG"),
    (dict(a=-1.0), "SS_ERR_INVALID_ARG"),
    (dict(a=float("inf")), "SS_ERR_INVALID_ARG"),
    (dict(kv=FAKE + 4), "SS_ERR_INVALID_ARG"),
    (dict(Hq=65), "SS_ERR_UNSUPPORTED"),
    (dict(d_rope=32), "SS_ERR_UNSUPPORTED"),
    (dict(S=4, ws=None), "SS_ERR_WORKSPACE"),
])
def test_mla_paged_decode_rejects_before_launch(capi, kw, expect):
    args = dict(kv=FAKE, table=FAKE, lens=FAKE, Hq=16, num_pages=10, max_pages=4, d_rope=64,
                a=1.0, S=1, ws=FAKE, ws_bytes=1 << 30)
    args.update(kw)
    st = capi.ss_attn_mla_decode_paged(FAKE, args["kv"], args["table"], args["lens"], FAKE, 2,
                                       args["Hq"], args["num_pages"], args["max_pages"], 512,
                                       args["d_rope"], 0.07, args["a"], args["S"], None,
                                       args["ws"], args["ws_bytes"], stream=0)
    assert st == getattr(capi, expect)


def test_mla_calibration_problem_checks(capi):
    """A latent-attention calibration problem must have one KV head and the
    576-entry key width; checked before anything runs."""
    cnt = FAKE
    for Hkv, d in ((2, 576), (1, 128)):
        prob = capi.ss_problem(capi.SS_MLA_DECODE, FAKE, FAKE, None, 2, 16, Hkv, 1, 1000, d, 0.07,
                               0, 1, cnt, 0)
        st, _, _ = capi.ss_calibrate(prob, 0.5)
        assert st == capi.SS_ERR_UNSUPPORTED


def test_struct_layouts_match_the_header(capi, tmp_path):
    """ctypes mirrors of the C structs have the C compiler's sizes and offsets."""
    src = tmp_path / "sz.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "ssattn.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu %zu %zu %zu\\n", sizeof(ss_debug_opts), sizeof(ss_problem),\n'
        "         offsetof(ss_debug_opts, fault_inject), offsetof(ss_debug_opts, prefill_kernel),\n"
        "         offsetof(ss_problem, skip_counts),\n"
        "         offsetof(ss_problem, stream), offsetof(ss_problem, fault_inject));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)], text=True).split()]
    want = [ctypes.sizeof(capi.ss_debug_opts), ctypes.sizeof(capi.ss_problem),
            capi.ss_debug_opts.fault_inject.offset, capi.ss_debug_opts.prefill_kernel.offset,
            capi.ss_problem.skip_counts.offset,
            capi.ss_problem.stream.offset, capi.ss_problem.fault_inject.offset]
    assert got == want


def test_workspace_size(capi):
    assert capi.ss_attn_decode_workspace_size(64, 32, 128, 1) == 0
    assert capi.ss_attn_decode_workspace_size(64, 32, 128, 8) == 64 * 32 * 8 * 130 * 4
    assert capi.ss_attn_mla_decode_workspace_size(64, 16, 512, 1) == 0
    assert capi.ss_attn_mla_decode_workspace_size(64, 16, 512, 16) == 64 * 16 * 16 * 514 * 4


def test_static_scratch_size_matches_the_library(capi):
    """The binding's copy of SS_DECODE_STATIC_SCRATCH_BYTES equals the size of
    the array compiled into the library, and the header's define."""
    src = open(HEADER).read()
    m = re.search(r"#define SS_DECODE_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", src)
    assert m, "define not found"
    header = int(m.group(1)) << int(m.group(2))
    assert capi.ss_decode_static_scratch_bytes() == header == capi.SS_DECODE_STATIC_SCRATCH_BYTES


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "block_sparse_attention_sm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.h" not in text, f


def test_rebuild_is_keyed_on_the_sources(capi):
    """The library is rebuilt when its recorded source hash differs from the
    tree's (a library built from other sources is never trusted because of
    its file time)."""
    from block_sparse_attention_sm_gb300 import builder

    assert not builder._stale()
    saved = open(builder.STAMP).read()
    try:
        with open(builder.STAMP, "w") as f:
            f.write("0" * 64 + "\n")
        assert builder._stale()
    finally:
        with open(builder.STAMP, "w") as f:
            f.write(saved)
    assert not builder._stale()
    assert builder._stale(["-DSOMETHING_ELSE"])  # other flags, other library
