"""Host-side tests of libra.so: exports, argument checks, planner, layout maps.

No GPU is needed: the planner's tile counts and the layout maps are pure host
code, checked bit for bit against the oracle.  Nothing here launches a kernel.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from tests.conftest import ROOT

ra = pytest.importorskip("context_ring_attention_gb300")


@pytest.fixture(scope="module")
def lib():
    from context_ring_attention_gb300 import build
    if not os.path.exists(ra.library_path()):
        build.build()
    return ra.load_library()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "ra.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert set(names) == set(ra.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_status_names_match_header():
    with open(os.path.join(ROOT, "include", "ra.h")) as f:
        text = f.read()
    codes = {int(v): n for n, v in re.findall(r"\b(RA_(?:OK|ERR_[A-Z_]+))\s*=\s*(\d+)", text)}
    assert codes == ra._STATUS


def test_debug_build_exports_the_same_symbols():
    from context_ring_attention_gb300 import build
    if not os.path.exists(build.LIB_DEBUG):
        build.build(debug=True)
    dbg = ctypes.CDLL(build.LIB_DEBUG)
    for n in _declared_symbols():
        assert hasattr(dbg, n), n


def test_status_word_decoding(tmp_path):
    """The status word -> error mapping that ra_sync_status and ra_fwd_static_status
    share: the bounds bit wins and reports its sites; otherwise a timeout."""
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if gxx is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    src = tmp_path / "decode.cpp"
    src.write_text(
        '#include "ra_internal.h"\n'
        "int main() {\n"
        "  char m[200];\n"
        "  if (ra::status_word_error(ra::kStatusTimeoutMma, m, sizeof m) != RA_ERR_TIMEOUT) return 1;\n"
        "  if (ra::status_word_error(ra::kStatusBounds | (0x2Au << 8), m, sizeof m) != RA_ERR_BOUNDS) return 2;\n"
        "  if (std::string(m).find(\"0x2a\") == std::string::npos) return 3;\n"
        "  if (ra::status_word_error(ra::kStatusBounds | ra::kStatusTimeoutSoftmax, m, sizeof m) != RA_ERR_BOUNDS)"
        " return 4;\n"
        "  return 0;\n"
        "}\n")
    exe = tmp_path / "decode"
    csrc = os.path.join(ROOT, "context_ring_attention_gb300", "csrc")
    res = subprocess.run([gxx, "-std=c++17", "-include", "string", "-I", cuda_inc, "-I", csrc, "-I",
                          os.path.join(ROOT, "include"), str(src), "-o", str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    assert subprocess.run([str(exe)]).returncode == 0


def test_library_variant_selects_the_debug_build(monkeypatch):
    monkeypatch.setenv("RA_LIBRARY_VARIANT", "debug")
    assert os.path.basename(ra.library_path()) == "libra_debug.so"
    monkeypatch.delenv("RA_LIBRARY_VARIANT")
    assert os.path.basename(ra.library_path()) == "libra.so"


def test_no_device_plan_refuses_fwd(lib):
    pytest.importorskip("torch")
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    plan = ra.ra_plan(1, 256, 2, 2, 128, 2, "contiguous", True, "bf16")
    buf = ctypes.create_string_buffer(4096 + 16)
    addr = (ctypes.addressof(buf) + 15) & ~15
    st = lib.ra_fwd(plan.handle, addr, addr, addr, addr, None, None, None, None)
    assert st == 5   # RA_ERR_NO_DEVICE
    assert "without a CUDA device" in ra.ra_last_error()
    word = ctypes.c_uint32(7)
    assert lib.ra_wait_selftest(ctypes.addressof(word)) == 5
    assert word.value == 7


@pytest.mark.parametrize("kw,status", [
    (dict(seq=100, n_shards=8), 1),                                  # uneven shards
    (dict(seq=20, n_shards=4, layout="zigzag"), 1),                 # zigzag needs 2N | S
    (dict(heads_q=6, heads_kv=4), 1),                               # Hq % Hkv
    (dict(head_dim=64), 2),                                         # bf16 needs d == 128
    (dict(dtype="f32", head_dim=256), 2),                           # f32 d <= 128
    (dict(batch=0), 1),
    (dict(scale=-1.0), 1),
    # planner limits: N^2 x query tiles above 2^30; bf16 work lists above 2^27 entries
    (dict(seq=32767 * 1024, n_shards=32767, heads_q=1, heads_kv=1), 2),
    (dict(seq=4096 * 1024, n_shards=4096, heads_q=2, heads_kv=1), 2),
    # B * Hq * S rows must fit the kernels' 32-bit row coordinates: 32 x 2^26 = 2^31
    (dict(seq=1 << 26, heads_q=32, heads_kv=8), 2),
    (dict(seq=1 << 26, heads_q=32, heads_kv=8, dtype="f32", head_dim=64), 2),
])
def test_plan_rejects(lib, kw, status):
    args = dict(batch=1, seq=1024, heads_q=4, heads_kv=2, head_dim=128, n_shards=8, layout="contiguous",
                causal=True, dtype="bf16", scale=0.0)
    args.update(kw)
    with pytest.raises(ra.RaError) as ei:
        ra.ra_plan(**args)
    assert ei.value.status == status


def test_null_arguments(lib):
    assert lib.ra_plan(None, None) == 1
    assert lib.ra_plan_tile_counts(None, None, None, None) == 1
    assert lib.ra_merge_partials(0, 1, 1, None, None, None, 0, None, None) == 1
    assert lib.ra_layout_perm(0, 8, 2, 0, 1, 4, None, None, None) == 1
    assert lib.ra_layout_index(0, 8, 3, None) == 1
    assert lib.ra_plan_destroy(None) == 0
    assert lib.ra_wait_selftest(None) == 1


def test_layout_perm_rejects_overlap_and_alignment(lib):
    buf = ctypes.create_string_buffer(8192 + 32)
    a = (ctypes.addressof(buf) + 15) & ~15
    assert lib.ra_layout_perm(0, 16, 2, 0, 1, 4, a, a + 16, None) == 1      # overlap
    assert lib.ra_layout_perm(0, 16, 2, 0, 1, 4, a + 4, a + 4096, None) == 1  # misaligned
    assert lib.ra_layout_perm(0, 16, 2, 0, 1, 6, a, a + 4096, None) == 1     # row_bytes % 4
    assert lib.ra_layout_perm(0, 1 << 30, 2, 0, 1 << 40, 256, a, a + 4096, None) == 2  # size overflows


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("seq,n", [(12, 4), (96, 8), (4096, 32), (32768, 8), (1000, 10)])
def test_layout_index_matches_oracle(lib, layout, seq, n):
    if layout == "zigzag" and seq % (2 * n):
        pytest.skip("zigzag needs 2N | S")
    assert ra.ra_layout_index(layout, seq, n).tolist() == oracle.layout_positions(layout, seq, n).tolist()


CASES = [
    ("contiguous", 32768, 8), ("zigzag", 32768, 8), ("striped", 131072, 32), ("zigzag", 1048576, 8),
    ("contiguous", 1000, 4), ("striped", 1000, 4), ("zigzag", 1000, 4), ("striped", 96 * 8, 8),
    ("zigzag", 4 * 300, 2), ("contiguous", 12, 4), ("striped", 640, 5),
]


@pytest.mark.parametrize("layout,seq,n", CASES)
@pytest.mark.parametrize("causal", [True, False])
def test_tile_counts_match_oracle(lib, layout, seq, n, causal):
    plan = ra.ra_plan(1, seq, 4, 2, 128, n, layout, causal, "bf16")
    got = ra.ra_plan_tile_counts(plan)
    want = oracle.tile_counts(layout, seq, n, causal=causal, tile=128)
    for g, w in zip(got, want):
        assert g.tolist() == w.tolist()


def _random_problems(n_cases=60, seed=2024):
    """Seeded (layout, seq, n_shards, causal) draws: ragged shards, odd N, tiny and long shards."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n_cases:
        layout = ("contiguous", "striped", "zigzag")[rng.integers(3)]
        n = int(rng.integers(1, 17))
        unit = 2 * n if layout == "zigzag" else n
        seq = unit * int(rng.integers(1, 4096 // unit + 1))
        out.append((layout, seq, n, bool(rng.integers(2))))
    return out


@pytest.mark.parametrize("layout,seq,n,causal", _random_problems())
def test_tile_counts_match_oracle_random(lib, layout, seq, n, causal):
    plan = ra.ra_plan(1, seq, 2, 1, 128, n, layout, causal, "bf16")
    got = ra.ra_plan_tile_counts(plan)
    want = oracle.tile_counts(layout, seq, n, causal=causal, tile=128)
    for g, w in zip(got, want):
        assert g.tolist() == w.tolist()


@pytest.mark.parametrize("layout,seq,n,causal", _random_problems(seed=2025))
def test_layout_index_matches_oracle_random(lib, layout, seq, n, causal):
    assert ra.ra_layout_index(layout, seq, n).tolist() == oracle.layout_positions(layout, seq, n).tolist()


def test_tile_counts_seq32k_report():
    """The per-shard FULL/PARTIAL/SKIP table for 32768 tokens, 8 shards (reported by bench)."""
    for layout in ("contiguous", "zigzag"):
        plan = ra.ra_plan(1, 32768, 32, 8, 128, 8, layout, True, "bf16")
        full, part, skip = ra.ra_plan_tile_counts(plan)
        assert (full + part + skip).tolist() == [32 * 32 * 8] * 8
        if layout == "zigzag":
            assert len(set((full + part).tolist())) == 1          # exactly balanced
        else:
            assert (full + part).tolist() == sorted((full + part).tolist())


def test_ring_entry_points_check_arguments(lib):
    """Argument checks of ra_fwd_step / ra_ring_rotate / ra_ring_fwd (no launch)."""
    plan = ra.ra_plan(1, 1024, 4, 2, 128, 4, "zigzag", True, "bf16")
    a = 1 << 20                      # aligned fake device addresses: nothing is dereferenced
    kv = 1 * 2 * 1024 * 128 * 2      # bytes of one K or V
    h = plan.handle
    assert lib.ra_fwd_step(h, 4, a, a, a, a, a, None) == 1          # step out of range
    assert lib.ra_fwd_step(h, -1, a, a, a, a, a, None) == 1
    assert lib.ra_fwd_step(h, 0, None, a, a, a, a, None) == 1       # null q
    assert lib.ra_fwd_step(h, 0, a + 8, a, a, a, a, None) == 1      # misaligned
    assert lib.ra_fwd_step(None, 0, a, a, a, a, a, None) == 1
    assert lib.ra_ring_rotate(h, a, a + 4 * kv, None, a + 6 * kv, None) == 1       # null destination
    assert lib.ra_ring_rotate(h, a, a + 4 * kv, a + 16, a + 6 * kv, None) == 1     # dst overlaps src
    assert lib.ra_ring_rotate(h, a, a + 4 * kv, a + 2 * kv, a + 2 * kv + 16, None) == 1  # dsts overlap
    assert "overlaps" in ra.ra_last_error()
    k, v, kb, vb = a, a + kv, a + 2 * kv, a + 4 * kv
    assert lib.ra_ring_fwd(h, a, k, v, a, None, None, vb, a, a, None, None) == 1   # N > 1 needs k_buf
    assert lib.ra_ring_fwd(h, a, k, v, a, None, kb, kb + kv, a, a, None, None) == 1  # k_buf/v_buf overlap
    assert lib.ra_ring_fwd(h, a, k, v, a, None, k, vb, a, a, None, None) == 1      # k_buf overlaps K
    assert lib.ra_ring_fwd(h, a, k, v, None, None, kb, vb, a, a, None, None) == 1  # null o
    pytest.importorskip("torch")
    import torch
    if torch.cuda.is_available():
        return
    # well-formed calls on a plan without a device
    assert lib.ra_fwd_step(h, 3, a, a, a, a, a, None) == 5
    assert lib.ra_ring_rotate(h, a, a + 2 * kv, a + 4 * kv, a + 6 * kv, None) == 5
    assert lib.ra_ring_fwd(h, a, k, v, a, None, kb, vb, a, a, None, None) == 5


def test_plan_rejects_too_many_shards(lib):
    with pytest.raises(ra.RaError) as ei:
        ra.ra_plan(1, 65536, 1, 1, 128, 32768, "contiguous", False, "bf16")
    assert ei.value.status == 2


def test_bwd_checks_arguments(lib):
    plan = ra.ra_plan(1, 1024, 4, 2, 128, 4, "zigzag", True, "bf16")
    a = 1 << 20
    h = plan.handle
    assert lib.ra_bwd(h, a, a, a, a, a, a, a, a, a, None, None) == 1     # null scratch
    assert lib.ra_bwd(h, a, a, a, a, a, a, a, a, a + 4, a, None) == 1    # misaligned dv
    assert lib.ra_bwd(None, a, a, a, a, a, a, a, a, a, a, None) == 1
    pytest.importorskip("torch")
    import torch
    if not torch.cuda.is_available():
        assert lib.ra_bwd(h, a, a, a, a, a, a, a, a, a, a, None) == 5


def test_bwd_scratch_size(lib):
    # 64-row blocks of every (batch, query head, shard), 128 floats each
    plan = ra.ra_plan(2, 900, 4, 2, 128, 3, "contiguous", True, "bf16")
    assert ra.ra_bwd_scratch_size(plan) == 2 * 4 * 3 * 5 * 128 * 4   # 300 rows per shard -> 5 blocks
    assert lib.ra_bwd_scratch_size(None, None) == 1


def test_binding_buffer_check():
    # the binding's check on caller buffers (shape, dtype, contiguity, device)
    torch = pytest.importorskip("torch")
    cpu = torch.device("cpu")
    with pytest.raises(ValueError):   # right shape, dtype and layout, but not on a CUDA device
        ra._need("t", torch.empty((2, 3, 4)), (2, 3, 4), torch.float32, cpu)
    for bad in (torch.empty((2, 3, 5)), torch.empty((2, 3, 4), dtype=torch.bfloat16),
                torch.empty((2, 4, 3)).transpose(1, 2), "not a tensor"):
        with pytest.raises(ValueError):
            ra._need("t", bad, (2, 3, 4), torch.float32, cpu)
    with pytest.raises(ValueError):
        ra._need("t", torch.empty((2, 3, 4)), (2, 3, 4), torch.float32, torch.device("cuda", 0))
    with pytest.raises(ValueError):   # a CPU tensor never reaches the library
        ra.ra_layout_perm(torch.empty((1, 1, 8, 4)), "contiguous", 2)


C_PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "ra.h"

int main(void) {
  ra_problem p = {1, 32768, 32, 8, 128, 8, RA_LAYOUT_ZIGZAG, 1, RA_DTYPE_BF16, 0.0f};
  ra_plan_t plan = NULL;
  if (ra_plan(&p, &plan) != RA_OK) {
    printf("plan: %s\n", ra_last_error());
    return 1;
  }
  int64_t full[8], partial[8], skip[8];
  if (ra_plan_tile_counts(plan, full, partial, skip) != RA_OK) return 2;
  for (int i = 0; i < 8; ++i) printf("%lld %lld %lld\n", (long long)full[i], (long long)partial[i], (long long)skip[i]);
  int64_t pos[16];
  if (ra_layout_index(RA_LAYOUT_ZIGZAG, 16, 4, pos) != RA_OK) return 3;
  for (int i = 0; i < 16; ++i) printf("%lld%c", (long long)pos[i], i == 15 ? '\n' : ' ');
  ra_problem bad = p;
  bad.seq = 100;
  ra_plan_t none = NULL;
  if (ra_plan(&bad, &none) != RA_ERR_INVALID_ARG || none != NULL) return 4;
  printf("%s\n", ra_last_error());
  return ra_plan_destroy(plan) == RA_OK ? 0 : 5;
}
"""


def test_plain_c_caller(lib, tmp_path):
    # the header compiles as C99 and the library links and runs from a C program
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(ra.library_path())
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), ra.library_path(), f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()
    want = oracle.tile_counts("zigzag", 32768, 8, causal=True)
    got = np.array([[int(x) for x in ln.split()] for ln in out[:8]]).T
    assert [g.tolist() for g in got] == [w.tolist() for w in want]
    assert [int(x) for x in out[8].split()] == oracle.layout_positions("zigzag", 16, 4).tolist()
    assert "multiple" in out[9] or "uneven" in out[9]
