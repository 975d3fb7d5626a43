"""The C ABI without a GPU: libfa.so loads, exports every entry point that
include/fa.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
LIB = os.path.join(ROOT, "exact_attention_qk_gb300", "libfa.so")


@pytest.fixture(scope="module")
def fa():
    if not os.path.exists(LIB):
        from exact_attention_qk_gb300 import build
        build.build(selftest=False)
    import torch  # noqa: F401  (provides the CUDA runtime the library links)
    from exact_attention_qk_gb300 import fa as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["fa_fwd", "fa_fwd_splitkv", "fa_combine", "fa_workspace_size", "fa_num_splits",
              "fa_split_len", "fa_get_status", "fa_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(fa):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (fa_[a-z_0-9]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = fa.lib()
    for n in declared_functions():
        assert hasattr(lib, n)


def test_struct_layout_matches_header(fa, tmp_path):
    """Compile a C probe against include/fa.h and compare every field offset."""
    fields = [f[0] for f in fa.FwdArgs._fields_]
    src = tmp_path / "probe.c"
    body = "\n".join(f'  printf("%s %zu\\n", "{n}", offsetof(fa_fwd_args, {n}));' for n in fields)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "fa.h"\nint main(void){\n'
                   '  printf("sizeof %zu\\n", sizeof(fa_fwd_args));\n' + body + "\n  return 0;\n}\n")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    assert int(got["sizeof"]) == ctypes.sizeof(fa.FwdArgs)
    for n in fields:
        assert int(got[n]) == getattr(fa.FwdArgs, n).offset, n
    assert fa.fa_abi_version() == 202


def _args(fa, **over):
    a = fa.FwdArgs()
    a.q, a.k, a.v, a.out = 0x10000, 0x20000, 0x30000, 0x40000
    a.batch, a.seqlen_q, a.seqlen_k = 2, 300, 300
    a.num_heads_q, a.num_heads_kv, a.head_dim_qk, a.head_dim_v = 8, 2, 128, 128
    a.q_batch_stride, a.q_row_stride, a.q_head_stride = 300 * 8 * 128, 8 * 128, 128
    a.k_batch_stride, a.k_row_stride, a.k_head_stride = 300 * 2 * 128, 2 * 128, 128
    a.v_batch_stride, a.v_row_stride, a.v_head_stride = 300 * 2 * 128, 2 * 128, 128
    a.o_batch_stride, a.o_row_stride, a.o_head_stride = 300 * 8 * 128, 8 * 128, 128
    a.window_left, a.window_right = -1, -1
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(num_heads_q=6, num_heads_kv=4), 1),            # Hq % Hkv
    (dict(head_dim_qk=264), 1),                           # > 256
    (dict(head_dim_qk=100), 1),                           # not a multiple of 8
    (dict(head_dim_qk=96, head_dim_v=96), 2),             # legal but not compiled
    (dict(head_dim_qk=128, head_dim_v=64), 2),
    (dict(window_left=-2), 1),
    (dict(num_splits=257), 1),
    (dict(batch=-1), 1),
    (dict(q=0x10008), 3),                                 # 8-byte aligned only
    (dict(k_row_stride=2 * 128 + 4), 3),                  # stride not a multiple of 8 elements
    (dict(out=0), 1),
    (dict(q=0), 1),
])
def test_rejections_before_launch(fa, over, code):
    a = _args(fa, **over)
    assert fa.lib().fa_fwd(ctypes.byref(a), None, 0, None) == code


def test_varlen_needs_both_cu_seqlens(fa):
    a = _args(fa, cu_seqlens_q=0x50000)
    assert fa.lib().fa_fwd(ctypes.byref(a), None, 0, None) == 2


def test_empty_problem_is_a_no_op(fa):
    a = _args(fa, batch=0)
    assert fa.lib().fa_fwd(ctypes.byref(a), None, 0, None) == 0
    a = _args(fa, seqlen_q=0)
    assert fa.lib().fa_fwd(ctypes.byref(a), None, 0, None) == 0


def test_combine_rejections(fa):
    L = fa.lib()
    assert L.fa_combine(0x1000, 0x2000, 0, 1, 1, 1, 128, None, 0, 0x3000, 0, 0, 0, None, None) == 1
    assert L.fa_combine(0x1000, 0x2000, 257, 1, 1, 1, 128, None, 0, 0x3000, 0, 0, 0, None, None) == 1
    assert L.fa_combine(0x1000, 0x2000, 2, 1, 1, 1, 96, None, 0, 0x3000, 0, 0, 0, None, None) == 2
    assert L.fa_combine(0x1008, 0x2000, 2, 1, 1, 1, 128, None, 0, 0x3000, 128, 128, 128, None, None) == 3
    assert L.fa_combine(0x1000, 0x2000, 2, 0, 1, 1, 128, None, 0, 0x3000, 0, 0, 0, None, None) == 0


def test_split_policy(fa):
    # decode shape of the benchmark: Kmax 16384 -> 8 splits of 2048 keys
    a = _args(fa, batch=64, seqlen_q=1, seqlen_k=16384, num_heads_q=32, num_heads_kv=8)
    assert fa.fa_num_splits(a, 152) == 8
    assert fa.fa_split_len(a, 8) == 2048
    assert fa.fa_split_len(a, 3) == 64 * -(-(-(-16384 // 3)) // 64)
    # few units: more splits to fill the SMs
    a = _args(fa, batch=1, seqlen_q=1, seqlen_k=16384, num_heads_q=8, num_heads_kv=8)
    assert fa.fa_num_splits(a, 152) == 32
    # a prefill grid that fills more than half of the SMs, or has too few key
    # blocks to split (300 keys: 3 blocks), is not split
    a = _args(fa)
    assert fa.fa_num_splits(a, 152) == 1
    # the count fa_fwd would choose with num_splits == 0, whatever the field holds
    a = _args(fa, num_splits=5)
    assert fa.fa_num_splits(a, 152) == 1


def _batched(fa, B, sq, sk, hq, hkv, d=128, **over):
    a = _args(fa, batch=B, seqlen_q=sq, seqlen_k=sk, num_heads_q=hq, num_heads_kv=hkv, head_dim_qk=d, head_dim_v=d)
    a.q_batch_stride, a.q_row_stride, a.q_head_stride = sq * hq * d, hq * d, d
    a.o_batch_stride, a.o_row_stride, a.o_head_stride = sq * hq * d, hq * d, d
    a.k_batch_stride, a.k_row_stride, a.k_head_stride = sk * hkv * d, hkv * d, d
    a.v_batch_stride, a.v_row_stride, a.v_head_stride = sk * hkv * d, hkv * d, d
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_prefill_split_policy(fa):
    # 8 tiles (one 256-row tile per head) against 64 key blocks on 152 SMs:
    # min(152 // 8, 64 // 4, 32) = 16 splits of 4 blocks
    assert fa.fa_num_splits(_batched(fa, 1, 256, 8192, 8, 8), 152) == 16
    # one request's chunk: 32 unpacked tiles (256 rows are too many to pack), 128 key blocks
    assert fa.fa_num_splits(_batched(fa, 1, 256, 16384, 32, 8), 152) == 4
    # pack-GQA: 100 rows x 8 heads = 4 packed tiles per KV head, 4 KV heads = 16
    # tiles; 32 key blocks: min(9, 8, 32) = 8 -> 4 blocks per split -> 8
    assert fa.fa_num_splits(_batched(fa, 1, 100, 4096, 32, 4), 152) == 8
    # the chunked-prefill workload fills 128 of 152 SMs: not split
    assert fa.fa_num_splits(_batched(fa, 8, 128, 8192, 32, 4), 152) == 1
    # the split count shrinks so that no split is empty: 10 blocks, at most
    # 152 // 8 = 19 and 10 // 4 = 2 splits -> 2 of 5 blocks
    assert fa.fa_num_splits(_batched(fa, 1, 256, 1280, 8, 8), 152) == 2
    # fp8 caches stay on the decode kernel, unsplit at prefill shapes
    assert fa.fa_num_splits(_batched(fa, 1, 256, 8192, 8, 8, kv_format=1), 152) == 1
    # more SMs, more splits (capped at 32)
    assert fa.fa_num_splits(_batched(fa, 1, 256, 65536, 2, 2), 152) == 32


def test_status_strings(fa):
    for c in range(8):
        assert fa.fa_status_string(c)
    assert "unknown" in fa.fa_status_string(99)


@pytest.mark.parametrize("over,code", [
    (dict(page_table=0x50000, max_pages_per_seq=3, page_size=128, num_pages=6), 2),
    (dict(kv_format=1), 2),                               # fp8 cache
    (dict(head_dim_qk=256, head_dim_v=128), 2),           # a forward-only head-dim pair
    (dict(num_heads_q=6, num_heads_kv=4), 1),
    (dict(out=0), 1),
    (dict(lse=0), 1),                                     # the forward's LSE is an input
])
def test_backward_rejections_before_launch(fa, over, code):
    a = _args(fa, **over)
    if "lse" not in over:
        a.lse = 0x70000
    assert fa.lib().fa_bwd(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None) == code


@pytest.mark.parametrize("dk,dv", [(192, 128), (256, 256)])
def test_backward_accepts_large_head_dims(fa, dk, dv):
    # served; the call gets as far as the workspace check
    a = _args(fa, lse=0x70000, head_dim_qk=dk, head_dim_v=dv)
    assert fa.lib().fa_bwd(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None) == 4


def test_backward_accepts_seqused_k(fa):
    # seqused_k is served (the TAIL kernels); the call gets as far as the workspace check
    a = _args(fa, lse=0x70000, seqused_k=0x50000)
    assert fa.lib().fa_bwd(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None) == 4


def test_backward_workspace(fa):
    a = _args(fa, lse=0x70000)
    # lse2 and D for 2 x 8 heads x 384 padded rows, 256-byte aligned
    assert fa.fa_bwd_workspace_size(a) == 2 * 2 * 8 * 384 * 4
    assert fa.lib().fa_bwd(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None) == 4
    assert fa.lib().fa_bwd(ctypes.byref(a), 0x80008, 0x90000, 0xA0000, 0xB0000, None, 0, None) == 3
    # (192, 128) and (256, 256) are served (two dK/dV passes); pairs the forward lacks are not
    assert fa.fa_bwd_workspace_size(_args(fa, head_dim_qk=192, head_dim_v=128)) == 2 * 2 * 8 * 384 * 4
    assert fa.fa_bwd_workspace_size(_args(fa, head_dim_qk=256, head_dim_v=256)) == 2 * 2 * 8 * 384 * 4
    assert fa.fa_bwd_workspace_size(_args(fa, head_dim_qk=256, head_dim_v=128)) == 0
    assert fa.lib().fa_bwd(ctypes.byref(_args(fa, batch=0)), 0, 0, 0, 0, None, 0, None) == 0


def test_backward_varlen_workspace(fa):
    # packed varlen: per q head, total_q + 132 rows per sequence + 4, rounded up to 32 rows
    a = _args(fa, lse=0x70000, cu_seqlens_q=0x50000, cu_seqlens_k=0x60000, total_q=600, total_k=600,
              max_seqlen_q=300, max_seqlen_k=300)
    rows = -(-(600 + 132 * 2 + 4) // 32) * 32
    per = -(-(8 * rows * 4) // 256) * 256
    assert fa.fa_bwd_workspace_size(a) == 2 * per
    # accepted: the next check is the missing workspace
    assert fa.lib().fa_bwd(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None) == 4


def test_bwd_two_streams_needs_the_callers_stream_and_events(fa):
    a = _args(fa, lse=0x70000)
    call = fa.lib().fa_bwd_two_streams
    # a missing second stream or event, or the second stream equal to the first: refused before any launch
    assert call(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None, None, 0x1, 0x2) == 1
    assert call(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None, 0x5, None, 0x2) == 1
    assert call(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, 0x5, 0x5, 0x1, 0x2) == 1
    # otherwise the same checks as fa_bwd (workspace missing)
    assert call(ctypes.byref(a), 0x80000, 0x90000, 0xA0000, 0xB0000, None, 0, None, 0x5, 0x1, 0x2) == 4
