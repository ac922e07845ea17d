"""The C ABI without a GPU: the library loads, exports every function the
header declares, its host helpers agree with the oracle, and argument checks
reject bad calls before any launch (host-side fault handling)."""
import ctypes
import os
import re

import numpy as np
import pytest

from compressed_kv_sparse_gb300 import lib
from oracle import rope, schedule

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "ds4a.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(lib.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return lib.load()


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^[a-z_0-9 \*]*?\b(ds4a_[a-z_0-9]+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(L):
    names = declared()
    assert set(names) == set(lib.EXPORTS)
    for n in names:
        assert hasattr(L, n), n
        assert n in lib.EXPORTS, f"binding does not declare {n}"


def test_schedule_and_chunk_cap_match_oracle(L):
    for variant in (0, 1):
        for il in range(64):
            assert L.ds4a_layer_compress_ratio(variant, il) == \
                schedule.layer_compress_ratio(variant, il)
    for n in (1, 4096, 4097, 28672, 100000):
        assert L.ds4a_prefill_chunk_cap(n) == schedule.prefill_chunk_cap(n)


def test_cache_bytes_match_oracle_and_page(L):
    ctx = 1 << 20
    tot = sum(L.ds4a_cache_bytes(schedule.layer_compress_ratio(1, il), 512, 128, ctx, 1, 2)
              for il in range(61))
    assert round(tot / 2**30, 2) == 9.62
    for ratio in (0, 4, 128):
        for c in (5, 127, 65536, 131072):
            assert L.ds4a_cache_bytes(ratio, 512, 128, c, 3, 2) == \
                schedule.kv_cache_bytes(ratio, 512, 128, c, 3, 2)


def test_rope_table_bitwise_equal_to_oracle(L):
    for base, n_rot in ((10000.0, 64), (160000.0, 64), (160000.0, 32)):
        n_pos = 2000
        c = np.empty((n_pos, n_rot // 2), np.float32)
        s = np.empty((n_pos, n_rot // 2), np.float32)
        assert L.ds4a_rope_table(base, n_rot, n_pos, c.ctypes.data, s.ctypes.data) == 0
        pos = np.concatenate([np.arange(n_pos)])
        oc, os_ = rope.rope_coeffs(pos, base, n_rot)
        assert np.array_equal(c, oc) and np.array_equal(s, os_)
    # large positions (the 131,072-token workloads)
    n_pos = 131073
    c = np.empty((n_pos, 32), np.float32)
    s = np.empty((n_pos, 32), np.float32)
    L.ds4a_rope_table(160000.0, 64, n_pos, c.ctypes.data, s.ctypes.data)
    idx = np.array([65535, 65536, 100003, 131071, 131072])
    oc, os_ = rope.rope_coeffs(idx, 160000.0, 64)
    assert np.array_equal(c[idx], oc) and np.array_equal(s[idx], os_)


def test_status_strings(L):
    for st in range(0, -9, -1):
        assert L.ds4a_status_string(st).decode() == lib.STATUS[st]


def _fake_cache(ratio=4, n_tokens=10, dtype=lib.DS4A_BF16):
    """A struct with non-NULL fake device pointers: only ever read by the host
    checks below, which return before touching them."""
    fake = 0x1000
    return lib.LayerCacheC(ratio=ratio, head_dim=512, n_rot=64, index_dim=128, index_rot=64,
                           batch=2, cap_raw=128, comp_cap=16, dtype=dtype, n_tokens=n_tokens,
                           raw_kv=fake, attn_comp_kv=fake, attn_state_kv=fake,
                           attn_state_score=fake, index_comp_kv=fake, index_state_kv=fake,
                           index_state_score=fake, index_norm=fake, index_norm_max=fake,
                           rope_cos=fake, rope_sin=fake, index_rope_cos=fake,
                           index_rope_sin=fake, rope_max_pos=1000)


def test_cache_struct_layout_matches_header(tmp_path):
    """The binding's struct has the header's field offsets and size (a C
    program compiled against include/ds4a.h prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in lib.LayerCacheC._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "ds4a.h"\nint main(void){'
                   + "".join(f'printf("%zu ", offsetof(ds4a_layer_cache, {f}));' for f in fields)
                   + 'printf("%zu\\n", sizeof(ds4a_layer_cache));return 0;}\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    want = [getattr(lib.LayerCacheC, f).offset for f in fields] + [ctypes.sizeof(lib.LayerCacheC)]
    assert got == want


def test_argument_checks_reject_before_launch(L):
    fake = 0x1000
    c = _fake_cache()
    r = ctypes.byref(c)
    P = [fake] * 9
    # wrong position: the cache holds 10 tokens
    assert L.ds4a_compress_append(r, 9, 1, *P, None, None) == -4
    # capacity: 16 compressed rows hold 64 tokens of ratio 4
    assert L.ds4a_compress_append(r, 10, 60, *P, None, None) == -3
    # rope table too short
    c.comp_cap = 10**6
    assert L.ds4a_compress_append(r, 10, 991, *P, None, None) == -3
    c.comp_cap = 16
    # missing lane inputs
    assert L.ds4a_compress_append(r, 10, 1, fake, None, fake, fake, fake, fake, fake, fake, fake,
                                  None, None) == -1
    assert c.n_tokens == 10        # nothing advanced
    # bad dtype / ratio / shapes
    bad = _fake_cache(dtype=7)
    assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == -5
    bad = _fake_cache(ratio=8)
    assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == -1
    bad = _fake_cache()
    bad.n_rot = 1000
    assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == -2
    # a ratio-4 cache without its row norms; the norm rebuild on another ratio
    bad = _fake_cache()
    bad.index_norm = None
    assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == -1
    assert L.ds4a_index_norms(ctypes.byref(_fake_cache(ratio=128)), None) == -1
    # index: reads beyond the appended tokens, workspace too small, bad ratio
    assert L.ds4a_index_topk(r, 10, 1, fake, fake, 64, 512, fake, fake, 1 << 30, None) == -4
    assert L.ds4a_index_topk(r, 9, 1, fake, fake, 64, 512, fake, fake, 16, None) == -8
    assert L.ds4a_index_topk(r, 9, 1, fake, fake, 64, 0, fake, fake, 1 << 30, None) == -2
    c128 = _fake_cache(ratio=128)
    assert L.ds4a_index_topk(ctypes.byref(c128), 9, 1, fake, fake, 64, 512, fake, fake,
                             1 << 30, None) == -1
    # the no-allocation variant runs the same checks before its scratch-size
    # check: the same statuses, and nothing touches a device
    assert L.ds4a_index_topk_noalloc(ctypes.byref(c128), 9, 1, fake, fake, 64, 512, fake,
                                     None) == -1
    assert L.ds4a_index_topk_noalloc(r, 10, 1, fake, fake, 64, 512, fake, None) == -4
    assert L.ds4a_index_topk_noalloc(r, 9, 1, fake, fake, 64, 0, fake, None) == -2
    assert L.ds4a_index_topk_noalloc(r, 9, 1, None, fake, 64, 512, fake, None) == -1
    assert L.ds4a_index_topk_noalloc(None, 9, 1, fake, fake, 64, 512, fake, None) == -1
    # lane-selective append: empty or unknown lane set, a lane the layer lacks,
    # and the position check (n_tokens stays for the caller to set)
    assert L.ds4a_compress_append_lanes(r, 10, 1, 0, *P, None, None) == -1
    assert L.ds4a_compress_append_lanes(r, 10, 1, 8, *P, None, None) == -1
    assert L.ds4a_compress_append_lanes(ctypes.byref(_fake_cache(ratio=128)), 10, 1,
                                        lib.LANE_INDEX, *P, None, None) == -1
    assert L.ds4a_compress_append_lanes(ctypes.byref(_fake_cache(ratio=0)), 10, 1,
                                        lib.LANE_ATTN, *P, None, None) == -1
    assert L.ds4a_compress_append_lanes(r, 9, 1, lib.LANE_RAW, *P, None, None) == -4
    assert c.n_tokens == 10
    # paged cache: a table on a window-only layer, comp_cap not max_blocks rows
    # of 256 positions, no blocks
    bad = _fake_cache(ratio=0)
    bad.block_table, bad.max_blocks, bad.n_blocks = fake, 4, 8
    assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == -1
    bad = _fake_cache()
    bad.block_table, bad.max_blocks, bad.n_blocks = fake, 4, 8   # 4 blocks = 256 rows != 16
    assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == -2
    bad.max_blocks, bad.n_blocks = 1, 0
    assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == -1
    # per-sequence positions (ragged batches) take chunks as well as single
    # tokens: the calls check the call's pos0 against n_tokens as before
    rg = _fake_cache()
    rg.seq_pos = fake
    assert L.ds4a_compress_append(ctypes.byref(rg), 9, 2, *P, None, None) == -4
    assert L.ds4a_index_topk(ctypes.byref(rg), 9, 2, fake, fake, 64, 512, fake, fake, 1 << 30,
                             None) == -4
    assert L.ds4a_sparse_attn_prefill_chunk(ctypes.byref(rg), 7, 2, fake, 64, fake, fake, 512,
                                            0.1, fake, fake, 1 << 30, None) == -4
    assert L.ds4a_compress_append(ctypes.byref(rg), 9, 1, *P, None, None) == -4
    # step-8 flags: unknown bit, FP4 off ratio 4, FP4 with Di not a power of two,
    # FP8 on a window-only layer
    for ratio, q, dim, want in ((4, 4, 128, -1), (128, 2, 128, -1), (4, 2, 96, -2),
                                (0, 1, 128, -1)):
        bad = _fake_cache(ratio=ratio)
        bad.qat, bad.index_dim = q, dim
        assert L.ds4a_compress_append(ctypes.byref(bad), 10, 1, *P, None, None) == want
    ok = _fake_cache()
    ok.qat = lib.QAT_FP8_ATTN | lib.QAT_FP4_INDEX
    assert L.ds4a_compress_append(ctypes.byref(ok), 9, 1, *P, None, None) == -4  # past the flag check
    # attention: position, missing top-k on a ratio-4 layer, workspace
    assert L.ds4a_sparse_attn_decode(r, 8, fake, 64, fake, 512, 0.1, fake, fake, 1 << 30,
                                     None) == -4
    assert L.ds4a_sparse_attn_decode(r, 9, fake, 64, None, 512, 0.1, fake, fake, 1 << 30,
                                     None) == -1
    need = L.ds4a_workspace_bytes(lib.CALL_ATTN_DECODE, r, 1, 64, 512)
    assert need > 0
    assert L.ds4a_sparse_attn_decode(r, 9, fake, 64, fake, 512, 0.1, fake, fake, need - 1,
                                     None) == -8
    assert L.ds4a_sparse_attn_prefill_chunk(r, 0, 5, fake, 64, None, fake, 512, 0.1, fake,
                                            fake, 1 << 30, None) == -1
    assert L.ds4a_sparse_attn_prefill_chunk(r, 0, 5, fake, 64, fake, fake, 512, 0.1, fake,
                                            fake, 1 << 30, None) == -4
    assert L.ds4a_sparse_attn_decode(None, 9, fake, 64, fake, 512, 0.1, fake, fake, 1 << 30,
                                     None) == -1


def test_paged_cache_layout_helpers_on_cpu(L):
    """The binding's paged layout without a GPU: a history scattered into the
    pools through a block table (random order, a shared prefix) gathers back
    to the same logical rows, and the struct carries the table."""
    import torch
    B, max_blocks, n_blocks, D, rpb = 3, 5, 20, 16, 2      # ratio 128: 2 rows per block
    perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(0))
    table = perm[:B * max_blocks].reshape(B, max_blocks).to(torch.int32)
    table[1:, :2] = table[0, :2]                            # shared first two blocks
    rows = torch.randn(B, max_blocks * rpb, D)
    rows[1:, :2 * rpb] = rows[0, :2 * rpb]
    c = lib.LayerCache(ratio=128, head_dim=D, n_rot=8, batch=B, comp_cap=max_blocks * rpb,
                       dtype="f32", base=10000.0, rope_max_pos=16, device="cpu",
                       block_table=table, n_blocks=n_blocks)
    assert c.attn_comp_kv.shape == (n_blocks, rpb, D)
    c.load_state({"attn_comp_kv": rows}, 0)
    assert torch.equal(c.logical("attn_comp_kv"), rows)
    assert c.c.block_table == table.data_ptr() and c.c.max_blocks == max_blocks
    assert c.c.n_blocks == n_blocks and c.c.seq_pos is None
    pos = torch.tensor([5, 3, 9], dtype=torch.int32)
    c.set_seq_pos(pos)
    assert c.c.seq_pos == pos.data_ptr()


def test_plain_c_host_links_the_library(L, tmp_path):
    """A C program built with gcc against include/ds4a.h and linked to
    libds4a.so (no Python, no torch) gets the same host results as the
    oracle: the 61-layer Pro schedule's cache bytes at 1M tokens (the page's
    9.62 GiB), a rope coefficient and an argument check."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "host.c"
    src.write_text(r'''
#include <stdio.h>
#include "ds4a.h"
int main(void) {
  unsigned long long tot = 0;
  for (unsigned il = 0; il < 61; ++il)
    tot += ds4a_cache_bytes(ds4a_layer_compress_ratio(1, il), 512, 128, 1u << 20, 1, 2);
  float c[3 * 32], s[3 * 32];
  const int st = ds4a_rope_table(160000.0, 64, 3, c, s);
  const int bad = ds4a_rope_table(160000.0, 63, 3, c, s);
  printf("%llu %d %d %.9g %.9g %s\n", tot, st, bad, c[32 + 1], s[2 * 32 + 5],
         ds4a_status_string((ds4a_status)bad));
  return 0;
}
''')
    exe = tmp_path / "host"
    libdir = os.path.dirname(lib.LIB_PATH)
    subprocess.run([cc, "-I", os.path.join(root, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lds4a", "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    tot, st, bad = int(out[0]), int(out[1]), int(out[2])
    assert round(tot / 2**30, 2) == 9.62
    assert tot == sum(schedule.kv_cache_bytes(schedule.layer_compress_ratio(1, il), 512, 128,
                                              1 << 20, 1, 2) for il in range(61))
    ref_c, ref_s = rope.rope_coeffs(np.arange(3), 160000.0, 64)
    assert st == 0 and np.float32(float(out[3])) == ref_c[1, 1]   # %.9g round-trips fp32
    assert np.float32(float(out[4])) == ref_s[2, 5]
    assert bad == -1 and " ".join(out[5:]) == "invalid argument"


def test_wait_status_and_cluster_hooks_on_cpu(L):
    """The wait status read-back maps a nonzero error word to DS4A_ERR_TIMEOUT
    and returns the count (a host copy of the word, read in place); the
    argument checks of the status, self-test and cluster calls reject bad
    values before touching a device."""
    word = (ctypes.c_int32 * 64)()
    n = ctypes.c_uint32(99)
    assert L.ds4a_workspace_status(ctypes.addressof(word), 256, ctypes.byref(n)) == 0
    assert n.value == 0
    word[0] = 3
    assert L.ds4a_workspace_status(ctypes.addressof(word), 256, ctypes.byref(n)) == -7
    assert n.value == 3
    assert L.ds4a_workspace_status(ctypes.addressof(word), 256, None) == -7
    assert L.ds4a_status_string(-7) == b"device wait timed out"
    assert L.ds4a_workspace_status(None, 256, ctypes.byref(n)) == -8
    assert L.ds4a_workspace_status(ctypes.addressof(word), 3, ctypes.byref(n)) == -8
    assert L.ds4a_workspace_clear_status(None, 256, None) == -8
    assert L.ds4a_wait_selftest(None, 256, 1000, None) == -8
    assert L.ds4a_wait_selftest(ctypes.addressof(word), 256, 0, None) == -1
    assert L.ds4a_wait_selftest(ctypes.addressof(word), 256, 1000001, None) == -1
    assert L.ds4a_set_decode_cluster(17) == -1
    assert L.ds4a_decode_cluster_size(None, 64, 512) == 0
