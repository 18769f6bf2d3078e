"""The C-ABI library builds, loads and exports every symbol include/raattn.h declares;
host-side validation rejects bad arguments before anything is launched.  No GPU:
only calls that return before touching the device are made here."""
import ctypes
import os

import pytest

import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300 import build as ra_build


@pytest.fixture(scope="module")
def lib():
    ra_build.build()
    return ra.lib()


def test_header_declares_the_boundary():
    names = ra.exported_symbols()
    for want in ("ra_softmax_fwd", "ra_softmax_bwd", "ra_attention_fwd", "ra_attention_bwd",
                 "ra_attention_bwd_workspace_size", "ra_status_string", "ra_device_status",
                 "ra_set_wait_limit_ns"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in ra.exported_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(5):
        assert lib.ra_status_string(code).decode().startswith("RA_")
    assert b"unknown" in lib.ra_status_string(99)


def test_workspace_size(lib):
    # one 5 x 128-float constant block per (head, 128-row query tile) (at least the two
    # per-row float arrays of the CUDA-core path) + fp16 copies of Q, dO (N_Q rows) and
    # K, V (N_K rows), then the masked calls' two tile maps (live and full), each both ways
    # (per head ceil(N_Q/128) rows of ceil(ceil(N_K/128)/32) words, and the transpose), and
    # one int per row of either layout; each piece padded to 256 bytes
    assert lib.ra_attention_bwd_workspace_size(4, 16, 8192, 8192, 128) == \
        (4 * 16 * 64 * 5 * 128 * 4) + 4 * (4 * 16 * 8192 * 128 * 2) + 4 * (4 * 16 * 64 * 2 * 4) + 2 * (4 * 16 * 64 * 4)
    assert lib.ra_attention_bwd_workspace_size(1, 1, 3, 3, 64) == 2560 + 4 * 512 + 4 * 256 + 2 * 256
    # ragged N_Q: 1000 rows make 8 query tiles per head; 16 keys one key tile
    assert lib.ra_attention_bwd_workspace_size(8, 8, 1000, 16, 64) == \
        (64 * 8 * 2560) + 2 * (64 * 1000 * 64 * 2) + 2 * (64 * 16 * 64 * 2) + 2 * (2048 + 256) + 2048 + 256
    assert lib.ra_attention_bwd_workspace_size(0, 1, 3, 3, 64) == 0
    assert lib.ra_attention_bwd_workspace_size(1, 1, -3, 3, 64) == 0


FAKE = ctypes.c_void_p(1 << 20)       # never dereferenced: every call below fails validation first
MISALIGNED = ctypes.c_void_p((1 << 20) + 4)
NULL = None
S = ctypes.c_void_p(0)


def test_softmax_validation(lib):
    assert lib.ra_softmax_fwd(NULL, FAKE, 4, 4, 0, S) == 1
    assert lib.ra_softmax_fwd(FAKE, FAKE, 0, 4, 0, S) == 1
    assert lib.ra_softmax_fwd(FAKE, FAKE, 4, -1, 0, S) == 1
    assert lib.ra_softmax_fwd(FAKE, FAKE, 4, 4, 7, S) == 1
    assert lib.ra_softmax_fwd(FAKE, FAKE, 1 << 40, 1 << 30, 0, S) == 1    # overflow
    assert lib.ra_softmax_fwd(NULL, FAKE, 4, 4, 1, S) == 1                # bf16: validated like fp32
    assert lib.ra_softmax_bwd(FAKE, NULL, FAKE, FAKE, 4, 4, 0, S) == 1


def _fwd(lib, q=FAKE, o=FAKE, ws=FAKE, B=1, H=1, NQ=8, NK=8, D=64, in_dt=1, out_dt=0, scale=0.0):
    return lib.ra_attention_fwd(q, FAKE, FAKE, o, NULL, NULL, NULL, NULL, ws, B, H, NQ, NK, D, scale, 0,
                                in_dt, out_dt, S)


def test_attention_fwd_validation(lib):
    assert _fwd(lib, q=NULL) == 1
    assert _fwd(lib, B=0) == 1
    assert _fwd(lib, NK=0) == 1
    assert _fwd(lib, D=-64) == 1
    assert _fwd(lib, in_dt=5) == 1
    assert _fwd(lib, q=MISALIGNED) == 1
    assert _fwd(lib, B=1 << 16, H=1 << 16) == 1                      # B*H overflows int32
    assert _fwd(lib, scale=float("inf")) == 1
    assert _fwd(lib, D=48) == 2                                       # bf16 tensor-core path: D in {64, 128}
    assert _fwd(lib, D=256) == 2
    assert _fwd(lib, D=48, in_dt=0) == 2                              # fp32 path: D in {16, 32, 64, 128}
    assert _fwd(lib, ws=NULL) == 1                                    # bf16 needs the fp16 V workspace
    assert _fwd(lib, ws=MISALIGNED) == 1
    # the fp16 V copy, then the masked calls' two tile maps (live and full: ceil(N_Q / 128)
    # rows of ceil(ceil(N_K / 128) / 32) words per head) and one int per row, each padded to
    # 256 bytes
    assert lib.ra_attention_fwd_workspace_size(4, 16, 8192, 8192, 128) == \
        4 * 16 * 8192 * 128 * 2 + 2 * (4 * 16 * 64 * 2 * 4) + 4 * 16 * 64 * 4
    assert lib.ra_attention_fwd_workspace_size(1, 3, 300, 5000, 64) == (3 * 5000 * 64 * 2 + 255) // 256 * 256 + 768
    assert lib.ra_attention_fwd_workspace_size(1, 1, 3, 3, 64) == 512 + 768   # 384 V bytes, 4 bytes per map and row
    assert lib.ra_attention_fwd_workspace_size(1, 1, 3, 0, 64) == 0


def test_attention_bwd_validation(lib):
    args = [FAKE] * 12
    ok_sizes = [1, 1, 8, 8, 64, 0.0, 0, 1, 0, 0, S]
    args_null = list(args)
    args_null[5] = NULL                                               # row_m is required
    assert lib.ra_attention_bwd(*args_null, *ok_sizes) == 1
    args_mis = list(args)
    args_mis[11] = MISALIGNED                                         # workspace misaligned
    assert lib.ra_attention_bwd(*args_mis, *ok_sizes) == 1
    bad_d = list(ok_sizes)
    bad_d[4] = 96
    assert lib.ra_attention_bwd(*args, *bad_d) == 2


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(ra, "_lib", None)
    monkeypatch.setattr(ra, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        ra.lib()


def test_product_package_never_imports_the_oracle():
    pkg = os.path.dirname(ra.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh")):
                with open(os.path.join(root, f)) as fh:
                    text = fh.read()
                assert "import oracle" not in text and "from oracle" not in text, f


def _fwd_masked(lib, mask=FAKE, MB=1, MH=1, B=2, H=2, in_dt=1):
    return lib.ra_attention_fwd_masked(FAKE, FAKE, FAKE, FAKE, NULL, NULL, NULL, NULL, FAKE, B, H, 8, 8, 64, 0.0, 0,
                                       in_dt, 0, mask, MB, MH, S)


def test_attention_mask_validation(lib):
    # one 32-bit word per 32 columns, rounded up to whole 128-column tiles
    assert [lib.ra_attention_mask_words(n) for n in (0, 1, 128, 129, 8192)] == [0, 4, 4, 8, 256]
    assert _fwd_masked(lib, mask=NULL) == 1
    assert _fwd_masked(lib, mask=MISALIGNED) == 1
    assert _fwd_masked(lib, MB=3) == 1                                # MB must be 1 or B
    assert _fwd_masked(lib, MH=0) == 1
    assert _fwd_masked(lib, in_dt=0) == 2                             # masks on the bf16 path only
    bwd = [FAKE] * 12 + [2, 2, 8, 8, 64, 0.0, 0, 1, 0, 0]
    assert lib.ra_attention_bwd_masked(*bwd, FAKE, NULL, 1, 1, S) == 1  # the key-major copy is required
    assert lib.ra_attention_bwd_masked(*bwd, FAKE, FAKE, 1, 3, S) == 1
    assert lib.ra_attention_mask_pack(NULL, 1, 8, 8, FAKE, FAKE, S) == 1
    assert lib.ra_attention_mask_pack(FAKE, 1, 8, 8, NULL, NULL, S) == 1
    assert lib.ra_attention_mask_pack(FAKE, 0, 8, 8, FAKE, FAKE, S) == 1
    assert lib.ra_attention_mask_pack(FAKE, 1, 8, 8, MISALIGNED, NULL, S) == 1


def test_pack_attn_mask_rejects_bad_masks():
    import torch
    with pytest.raises(NotImplementedError):
        ra.pack_attn_mask(torch.zeros(4, 4), 1, 1, 4, 4)              # additive float masks are not supported
