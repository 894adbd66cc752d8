"""The C ABI without a GPU: the library loads, exports every declared entry point,
and rejects each kind of invalid argument with its own status before launching
anything.  Pointers here are fake addresses that the library only compares; no
call in this file reaches a kernel launch."""
import ctypes
import os
import re

import pytest

from head_latent_attention_rmsnorm_gb300 import build as mla_build
from head_latent_attention_rmsnorm_gb300 import mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mla_build.build()
    return mla.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert "mla_latent_attn_fwd" in names and "mla_lse_combine" in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_distinct(L):
    codes = list(mla.STATUS)
    strs = {mla.mla_status_string(c) for c in codes}
    assert len(strs) == len(codes)
    for c, name in mla.STATUS.items():
        assert mla.mla_status_string(c).startswith(name)


V3 = dict(n_heads=128, d_kv=512, d_nope=128, d_rope=64, d_v=128)
BASE = 0x7f0000000000


def fake(i, bytes_each=1 << 32):
    """A 256-byte aligned fake device address; distinct i never overlap."""
    return BASE + i * bytes_each


def prefill_args(**over):
    d = mla.dims(**V3)
    a = dict(dims=ctypes.byref(d), dtype=mla.MLA_BF16, B=1, s_q=2048, s_kv=16384, q_offset=14336, causal=1,
             head_begin=0, head_count=128, head_shard=16, q_nope=fake(1), q_pe=fake(2), c_kv=fake(3),
             k_pe=fake(4), w_kv_b=fake(5), rms_w=fake(6), out=fake(7), lse=fake(8), workspace=fake(9),
             workspace_bytes=1 << 31, stream=None)
    a.update(over)
    a["_d"] = d
    return a


def call_prefill(fn, a):
    keys = ["dims", "dtype", "B", "s_q", "s_kv", "q_offset", "causal", "head_begin", "head_count",
            "head_shard", "q_nope", "q_pe", "c_kv", "k_pe", "w_kv_b", "rms_w", "out", "lse", "workspace",
            "workspace_bytes", "stream"]
    return fn(*[a[k] for k in keys])


@pytest.mark.parametrize("fn", ["mla_latent_attn_fwd", "mla_absorbed_attn_fwd"])
@pytest.mark.parametrize("over,status", [
    (dict(q_nope=None), -1),
    (dict(lse=None), -1),
    (dict(workspace=None), -1),
    (dict(s_q=4096), -2),                     # causal rows beyond the latent
    (dict(head_begin=120, head_count=16), -2),
    (dict(head_begin=2 ** 31 - 1, head_count=1), -2),   # the head range's end past INT_MAX
    (dict(q_offset=-1), -2),
    (dict(dtype=7), -3),
    (dict(out=fake(7) + 8), -4),
    (dict(workspace_bytes=1024), -5),
    (dict(out=fake(1) + 4096), -9),           # out inside q_nope
    (dict(workspace=fake(3) + 256), -9),      # workspace over c_kv
])
def test_prefill_rejects(L, fn, over, status):
    a = prefill_args(**over)
    assert call_prefill(getattr(mla, fn), a) == status


def test_prefill_unsupported_dims(L):
    d = mla.dims(n_heads=4, d_kv=1024, d_nope=128, d_rope=64, d_v=128)
    a = prefill_args(dims=ctypes.byref(d), head_count=4, head_shard=4)
    assert call_prefill(mla.mla_absorbed_attn_fwd, a) == -6


def test_prefill_bad_dims(L):
    d = mla.dims(n_heads=4, d_kv=512, d_nope=128, d_rope=63, d_v=128)   # odd RoPE band
    a = prefill_args(dims=ctypes.byref(d), head_count=4)
    assert call_prefill(mla.mla_latent_attn_fwd, a) == -2
    assert call_prefill(mla.mla_latent_attn_fwd, prefill_args(dims=None)) == -1


def test_prefill_empty_is_noop(L):
    for over in (dict(B=0), dict(s_q=0), dict(head_count=0), dict(B=0, q_nope=None)):
        assert call_prefill(mla.mla_latent_attn_fwd, prefill_args(**over)) == 0


def test_workspace_queries(L):
    d = mla.dims(**V3)
    f = mla.mla_latent_attn_workspace
    w16 = f(ctypes.byref(d), mla.MLA_BF16, 1, 2048, 16384, 14336, 1, 128, 16)
    w128 = f(ctypes.byref(d), mla.MLA_BF16, 1, 2048, 16384, 14336, 1, 128, 128)
    assert 0 < w16 < w128
    # explicit per-shard K/V: 16 heads x 16384 keys x 256 x 2 bytes dominate
    assert w16 >= 16 * 16384 * 256 * 2
    wa = mla.mla_absorbed_attn_workspace(ctypes.byref(d), mla.MLA_BF16, 1, 2048, 16384, 14336, 1, 128, 16)
    assert wa > 0
    assert f(ctypes.byref(d), mla.MLA_BF16, 1, 4096, 16384, 14336, 1, 128, 16) == 0   # invalid -> 0
    wd = mla.mla_decode_workspace(ctypes.byref(d), mla.MLA_BF16, 64, 32768, 8)
    assert wd >= 8 * 64 * 128 * 512 * 4                                            # fp32 partials


def decode_args(**over):
    d = mla.dims(**V3)
    a = dict(dims=ctypes.byref(d), dtype=mla.MLA_BF16, B=64, kv_len=32768, n_splits=8, q_nope=fake(1),
             q_pe=fake(2), c_cache=fake(3), kpe_cache=fake(4), w_kv_b=fake(5), out=fake(6), lse=fake(7),
             part_out=None, part_lse=None, workspace=fake(8), workspace_bytes=1 << 31, stream=None)
    a.update(over)
    a["_d"] = d
    keys = ["dims", "dtype", "B", "kv_len", "n_splits", "q_nope", "q_pe", "c_cache", "kpe_cache", "w_kv_b",
            "out", "lse", "part_out", "part_lse", "workspace", "workspace_bytes", "stream"]
    return [a[k] for k in keys], a


@pytest.mark.parametrize("over,status", [
    (dict(c_cache=None), -1),
    (dict(part_out=fake(9)), -1),             # part_out without part_lse
    (dict(n_splits=0), -2),
    (dict(n_splits=300), -2),
    (dict(kv_len=0), -2),
    (dict(dtype=5), -3),
    (dict(lse=fake(7) + 4), -4),
    (dict(workspace_bytes=4096), -5),
    (dict(out=fake(3) + 1024), -9),
    (dict(B=0), 0),
])
def test_decode_rejects(L, over, status):
    args, keep = decode_args(**over)
    assert mla.mla_decode_splitkv(*args) == status


def tpla_args(**over):
    d = mla.dims(**V3)
    a = dict(dims=ctypes.byref(d), dtype=mla.MLA_BF16, B=64, kv_len=32768, n_splits=8, n_shards=2,
             q_nope=fake(1), q_pe=fake(2), c_cache=fake(3), kpe_cache=fake(4), w_kv_b=fake(5), out=fake(6),
             slse=fake(7), workspace=fake(8), workspace_bytes=1 << 32, stream=None)
    a.update(over)
    a["_d"] = d
    keys = ["dims", "dtype", "B", "kv_len", "n_splits", "n_shards", "q_nope", "q_pe", "c_cache", "kpe_cache",
            "w_kv_b", "out", "slse", "workspace", "workspace_bytes", "stream"]
    return [a[k] for k in keys], a


@pytest.mark.parametrize("over,status", [
    (dict(c_cache=None), -1),
    (dict(slse=None), -1),
    (dict(n_shards=0), -2),
    (dict(n_shards=3), -2),                   # 512 latent dims do not split into 3
    (dict(n_shards=32), -2),
    (dict(n_splits=0), -2),
    (dict(dtype=5), -3),
    (dict(slse=fake(7) + 4), -4),
    (dict(workspace_bytes=4096), -5),
    (dict(slse=fake(3) + 1024), -9),          # shard lse inside the cache
    (dict(B=0), 0),
])
def test_tpla_decode_rejects(L, over, status):
    args, keep = tpla_args(**over)
    assert mla.mla_tpla_decode(*args) == status


def test_tpla_workspace_grows_with_shards(L):
    d = mla.dims(**V3)
    w1 = mla.mla_tpla_decode_workspace(ctypes.byref(d), mla.MLA_BF16, 64, 32768, 8, 1)
    w2 = mla.mla_tpla_decode_workspace(ctypes.byref(d), mla.MLA_BF16, 64, 32768, 8, 2)
    assert w1 == mla.mla_decode_workspace(ctypes.byref(d), mla.MLA_BF16, 64, 32768, 8)
    # the partials double and the expanded query rows are added
    assert w2 - w1 >= 8 * 64 * 128 * 512 * 4
    assert mla.mla_tpla_decode_workspace(ctypes.byref(d), mla.MLA_BF16, 64, 32768, 8, 3) == 0


@pytest.mark.parametrize("args,status", [
    ((mla.MLA_BF16, 10, 512, 2, 1e-6, None, fake(2), fake(3)), -1),
    ((mla.MLA_BF16, 10, 512, 3, 1e-6, fake(1), fake(2), fake(3)), -2),
    ((mla.MLA_BF16, 10, 512, 0, 1e-6, fake(1), fake(2), fake(3)), -2),
    ((mla.MLA_BF16, -1, 512, 1, 1e-6, fake(1), fake(2), fake(3)), -2),
    ((mla.MLA_BF16, 10, 512, 1, -1.0, fake(1), fake(2), fake(3)), -2),
    ((9, 10, 512, 1, 1e-6, fake(1), fake(2), fake(3)), -3),
    ((mla.MLA_BF16, 10, 512, 1, 1e-6, fake(1), fake(2) + 2, fake(3)), -4),
    ((mla.MLA_BF16, 10, 512, 1, 1e-6, fake(1), fake(2), fake(1) + 4096), -9),
    ((mla.MLA_BF16, 0, 512, 1, 1e-6, fake(1), fake(2), fake(3)), 0),
])
def test_rmsnorm_rejects(L, args, status):
    assert mla.mla_rmsnorm(*args, None) == status


@pytest.mark.parametrize("over,status", [
    (dict(dy=None), -1), (dict(ws=None), -1), (dict(n_shards=3), -2), (dict(rows=-1), -2), (dict(dtype=4), -3),
    (dict(dw=fake(5) + 4), -4), (dict(ws_bytes=16), -5), (dict(dx=fake(1) + 64), -9), (dict(dw=fake(3) + 16), -9),
])
def test_rmsnorm_bwd_rejects(L, over, status):
    a = dict(dtype=mla.MLA_BF16, rows=1000, d=512, n_shards=2, eps=1e-6, x=fake(1), w=fake(2), dy=fake(3),
             dx=fake(4), dw=fake(5), ws=fake(6), ws_bytes=1 << 30, stream=None)
    a.update(over)
    assert mla.mla_rmsnorm_bwd(*a.values()) == status
    assert mla.mla_rmsnorm_bwd_workspace(mla.MLA_BF16, 1000, 512, 2) >= 1000 * 2 * 4


@pytest.mark.parametrize("args,status", [
    ((mla.MLA_F32, 0, 10, 8, fake(1), fake(2), fake(3), fake(4), None), -2),
    ((mla.MLA_F32, 4, 10, 8, None, fake(2), fake(3), fake(4), None), -1),
    ((9, 4, 10, 8, fake(1), fake(2), fake(3), fake(4), None), -3),
    ((mla.MLA_F32, 4, 10, 8, fake(1), fake(2), fake(3) + 4, fake(4), None), -4),
    ((mla.MLA_F32, 4, 10, 8, fake(1), fake(2), fake(1) + 64, fake(4), None), -9),
    ((mla.MLA_F32, 4, 0, 8, fake(1), fake(2), fake(3), fake(4), None), 0),
])
def test_combine_rejects(L, args, status):
    assert mla.mla_lse_combine(*args) == status


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(mla, "_lib", None)
    monkeypatch.setattr(mla, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        mla.lib()


@pytest.mark.parametrize("limit_us", [0, 100001, 1 << 31])
def test_selftest_wait_limit_checked_before_launch(L, limit_us):
    assert mla.mla_selftest_bounded_wait(limit_us, None) == -2


def test_backward_validates_before_launch(L):
    d = mla.dims(**V3)
    base = [ctypes.byref(d), mla.MLA_BF16, 1, 2048, 16384, 14336, 1, 0, 128, 16] + [fake(i) for i in range(1, 16)]
    ws = mla.mla_latent_attn_bwd_workspace(ctypes.byref(d), mla.MLA_BF16, 1, 2048, 16384, 14336, 1, 128, 16)
    assert ws > 0
    args = base + [fake(20), ws, None]
    bad = list(args)
    bad[10] = None                                        # q_nope
    assert mla.mla_latent_attn_bwd(*bad) == -1
    bad = list(args)
    bad[19] = fake(19) + 8                                # dq_nope misaligned
    assert mla.mla_latent_attn_bwd(*bad) == -4
    bad = list(args)
    bad[26] = ws - 1                                      # workspace too small
    assert mla.mla_latent_attn_bwd(*bad) == -5
    bad = list(args)
    bad[19] = fake(1)                                     # dq_nope over q_nope
    assert mla.mla_latent_attn_bwd(*bad) == -9
    d2 = mla.dims(n_heads=128, d_kv=64, d_nope=300, d_rope=16, d_v=32)
    assert mla.mla_latent_attn_bwd(ctypes.byref(d2), mla.MLA_F32, *args[2:]) == -6


C_PROGRAM = r"""
#include <stdio.h>
#include "mla.h"
int main(void) {
    mla_dims d = {128, 512, 128, 64, 128, 10000.0f, 1e-6f, 0.0f};
    /* workspace query (host arithmetic only) */
    printf("%zu\n", mla_latent_attn_workspace(&d, MLA_BF16, 1, 2048, 16384, 14336, 1, 128, 16));
    /* validation before any launch: missing pointers, then a causal call past its keys */
    printf("%d\n", (int)mla_latent_attn_fwd(&d, MLA_BF16, 1, 16, 64, 0, 1, 0, 128, 16, NULL, NULL, NULL, NULL,
                                            NULL, NULL, NULL, NULL, NULL, 0, NULL));
    printf("%d\n", (int)mla_decode_splitkv(&d, MLA_BF16, 1, 0, 1, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                           NULL, NULL, NULL, 0, NULL));
    /* an empty call is a no-op */
    printf("%d\n", (int)mla_latent_attn_fwd(&d, MLA_BF16, 0, 16, 64, 0, 1, 0, 128, 16, NULL, NULL, NULL, NULL,
                                            NULL, NULL, NULL, NULL, NULL, 0, NULL));
    printf("%s\n", mla_status_string(MLA_ERR_SHAPE));
    return 0;
}
"""


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_builds_and_links_as_plain_c_and_cpp(L, tmp_path, lang):
    """A program in plain C11 (and the same as C++17, through the header's extern "C"
    block) includes include/mla.h, links libmla.so and calls the ABI without Python."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text(C_PROGRAM)
    exe = tmp_path / "t"
    libdir = os.path.dirname(mla.LIB_PATH)
    std = ["-std=c11"] if lang == "c" else ["-std=c++17"]
    subprocess.check_call([cc] + std + ["-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                                        "-L", libdir, "-lmla", "-Wl,-rpath," + libdir, "-o", str(exe)])
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    d = mla.dims(**V3)
    assert int(lines[0]) == mla.mla_latent_attn_workspace(ctypes.byref(d), mla.MLA_BF16, 1, 2048, 16384, 14336, 1,
                                                          128, 16)
    assert lines[1:5] == ["-1", "-2", "0", mla.mla_status_string(-2)]
