"""The C ABI without a GPU: the library loads, exports every declared symbol, and its
host-only logic (routing table, keep threshold, argument validation) agrees with the
oracle / the header's contract.  No call here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

from lora_fine_tuning_gb300 import native
from oracle import lora_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(native.LIB_PATH):
        from lora_fine_tuning_gb300 import build
        build.build()
    return native.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lora.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:lora_status|size_t|void|int32_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)


def test_header_and_binding_agree():
    assert declared_functions() == native.EXPORTED


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(9):
        assert native.status_string(code)
    assert native.status_string(0) == "ok"


@pytest.mark.parametrize("p", [0.0, 0.05, 0.1, 0.25, 0.5, 0.9, 0.999])
def test_keep_threshold_matches_oracle(lib, p):
    assert native.keep_threshold(p) == O.dropout_threshold(float(np.float32(p)))


@pytest.mark.parametrize("p", [1.0, -0.5, float("nan")])
def test_keep_threshold_rejects(lib, p):
    with pytest.raises(native.LoraError):
        native.keep_threshold(p)


@pytest.mark.parametrize("m,segments,n_ad", [
    (700, [(0, 128, 1), (256, 256, 0), (512, 188, 3)], 4),
    (1024, [], 2),
    (128 * 40, [(128 * i, 128, i % 3) for i in range(0, 40, 2)], 3),
    (300, [(0, 300, 0)], 1),
])
def test_tile_table_matches_oracle(lib, m, segments, n_ad):
    assert native.tile_table(segments, n_ad, m) == O.tile_adapters(segments, m, n_ad).tolist()


@pytest.mark.parametrize("segments", [[(64, 128, 0)], [(0, 100, 0), (128, 128, 0)], [(0, 256, 0), (128, 128, 1)],
                                      [(0, 128, 5)], [(0, 1024, 0)]])
def test_tile_table_rejects_like_oracle(lib, segments):
    with pytest.raises(ValueError):
        O.row_adapters(segments, 512, 2)
    with pytest.raises(native.LoraError) as e:
        native.tile_table(segments, 2, 512)
    assert e.value.status == 8


def test_workspace_size_grows(lib):
    a = lib.lora_workspace_size(1024, 512, 512, 16, 1)
    b = lib.lora_workspace_size(2048, 512, 512, 16, 1)
    c = lib.lora_workspace_size(1024, 512, 512, 64, 4)
    assert 0 < a < b and a < c
    assert a % 256 == 0


def _fwd_status(lib, *, X=256, W=256, A=256, B=256, alpha=1.0, p=0.1, m=128, k=64, n=64, r=16, Y=256, S=256,
                ws=256, ws_bytes=1 << 30):
    return lib.lora_fwd(X, W, A, B, alpha, p, 0, m, k, n, r, Y, S, None, ws, ws_bytes, None)


def test_validation_codes_without_launching(lib):
    """Every check runs before any CUDA call, so these return on a machine with no GPU."""
    assert _fwd_status(lib, k=60) == 3          # k not a multiple of 8
    assert _fwd_status(lib, n=0) == 3           # empty n
    assert _fwd_status(lib, m=300000) == 3      # too many rows
    assert _fwd_status(lib, k=(1 << 24) + 8) == 3   # more features than the 32-bit counts allow
    assert _fwd_status(lib, n=(1 << 24) + 8) == 3
    assert _fwd_status(lib, r=12) == 1          # rank not a multiple of 8
    assert _fwd_status(lib, r=136) == 1         # rank above 128
    assert _fwd_status(lib, p=1.0) == 1         # p outside [0, 1)
    assert _fwd_status(lib, p=-0.1) == 1
    assert _fwd_status(lib, X=258) == 2         # misaligned pointer
    assert _fwd_status(lib, A=264) == 2
    assert _fwd_status(lib, ws=None) == 6       # no workspace
    assert _fwd_status(lib, ws=512 + 16) == 6   # workspace not 256-aligned
    assert _fwd_status(lib, ws_bytes=100) == 6  # workspace too small
    assert _fwd_status(lib, X=None) == 1


def test_multi_validation_codes(lib):
    ad = (native.LoraAdapter * 2)()
    for i in range(2):
        ad[i].rank, ad[i].alpha, ad[i].p, ad[i].A, ad[i].B = 16, 1.0, 0.1, 256, 256
    bad_seg = native.segments_array([(0, 128, 0), (64, 128, 1)])
    st = lib.multi_lora_fwd(256, 256, ad, 2, bad_seg, 2, 0, 512, 64, 64, 256, 256, None, 256, 1 << 30, None)
    assert st == 8
    unknown = native.segments_array([(0, 128, 7)])
    st = lib.multi_lora_fwd(256, 256, ad, 2, unknown, 1, 0, 512, 64, 64, 256, 256, None, 256, 1 << 30, None)
    assert st == 8
    # segments with no adapters at all
    st = lib.multi_lora_fwd(256, 256, ad, 0, unknown, 1, 0, 512, 64, 64, 256, 256, None, 256, 1 << 30, None)
    assert st == 8
    # the backward needs gradient buffers
    st = lib.multi_lora_bwd(256, 256, 256, ad, 2, native.segments_array([(0, 128, 0)]), 1, 0, 512, 64, 64, 256,
                            None, 256, 256, 1 << 30, None)
    assert st == 1
    # saved keep bits must be 16-byte aligned like every other buffer
    st = lib.lora_bwd(256, 256, 256, 256, 256, 256, 264, 1.0, 0.1, 0, 128, 64, 64, 16, 256, 256, 256, 256, 1 << 30,
                      None)
    assert st == 2


@pytest.mark.parametrize("seed", range(12))
def test_pack_greedy_matches_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(0, 400))
    lengths = np.clip(np.round(rng.lognormal(6.2, 0.6, size=n)), 1, 2048).astype(int).tolist()
    capacity = int(128 * rng.choice([16, 32, 64, 128]))
    got = native.pack_greedy(lengths, capacity)
    if n == 0:
        assert got == ([], [], 0)
        return
    assert got == O.greedy_pack(lengths, capacity)


def test_pack_greedy_rejects(lib):
    with pytest.raises(native.LoraError) as e:
        native.pack_greedy([300], 256)
    assert e.value.status == 3
    for lengths, cap in (([10], 100), ([0], 256), ([10], 0)):
        with pytest.raises(native.LoraError) as e:
            native.pack_greedy(lengths, cap)
        assert e.value.status == 1


def test_pack_microbatches_make_valid_segment_tables(lib):
    rng = np.random.default_rng(7)
    lengths = np.clip(np.round(rng.lognormal(6.2, 0.6, size=300)), 64, 2048).astype(int).tolist()
    adapters = rng.integers(0, 4, size=300).tolist()
    batches = native.pack_microbatches(lengths, adapters, 16384)
    seen = []
    for b in batches:
        # the segment table is accepted by the library's own router and by the oracle's
        assert native.tile_table(b["segments"], 4, 16384) == O.tile_adapters(b["segments"], 16384, 4).tolist()
        for (start, rows, a), i, v in zip(b["segments"], b["samples"], b["valid"]):
            assert a == adapters[i] and v == lengths[i] and rows == O.padded_rows(v)
        seen += b["samples"]
    assert sorted(seen) == list(range(300))


def test_dora_workspace_and_validation(lib):
    assert lib.dora_workspace_size(1024, 512, 512, 16) > lib.lora_workspace_size(1024, 512, 512, 16, 1)
    # null magnitude vector / misaligned pointers are rejected before any CUDA call
    st = lib.dora_fwd(256, 256, 256, 256, None, 256, 1.0, 0.1, 0, 128, 64, 64, 16, 256, 256, 256, None, 256,
                      1 << 30, None)
    assert st == 1
    st = lib.dora_fwd(256, 256, 256, 256, 260, 256, 1.0, 0.1, 0, 128, 64, 64, 16, 256, 256, 256, None, 256,
                      1 << 30, None)
    assert st == 2
    st = lib.dora_bwd(256, 256, 256, 256, 256, 256, None, 256, 256, 256, 1.0, 0.1, 0, 128, 64, 64, 16, 256, 256,
                      256, None, 256, 256, 1 << 30, None)
    assert st == 1


def test_deterministic_mode_setter_and_workspace(lib):
    """Mode 1 sizes a larger workspace (slot region; no device here: the 1024-CTA bound); other values are
    rejected and leave the mode unchanged."""
    base = lib.lora_workspace_size(8192, 4096, 14336, 16, 1)
    assert lib.lora_get_deterministic() == 0
    assert lib.lora_set_deterministic(2) == 1           # LORA_EINVAL
    assert lib.lora_get_deterministic() == 0
    assert lib.lora_set_deterministic(1) == 0
    try:
        det = lib.lora_workspace_size(8192, 4096, 14336, 16, 1)
    finally:
        assert lib.lora_set_deterministic(0) == 0
    # slots: (64 tiles + 1024 CTAs) x 128 rows x 16 floats, or (32 feature blocks + 1024) x 128 x 16, whichever
    # is larger, rounded up to 256 bytes
    assert det - base == (64 + 1024) * 128 * 16 * 4
    assert lib.lora_workspace_size(8192, 4096, 14336, 16, 1) == base
