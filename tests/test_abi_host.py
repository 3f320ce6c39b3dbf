"""Host-side checks of the C ABI, no GPU needed: the library builds and loads,
exports every symbol include/kvq.h declares, and its pure-host calls (sizes,
validation) behave as the header states."""

import ctypes
import os
import re

import pytest

from quantized_kv_cache_08_gb300 import _binding as B
from quantized_kv_cache_08_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return B.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert _declared() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
    # the exported names are C symbols (no C++ mangling)
    for name in _declared():
        ctypes.CDLL(B.LIB_PATH)[name]


def test_block_bytes(L):
    assert B.kvq_block_bytes(B.KVQ_Q8_0) == 34
    assert B.kvq_block_bytes(B.KVQ_Q5_1) == 24
    assert B.kvq_block_bytes(B.KVQ_FP8_E4M3) == 32
    assert B.kvq_block_bytes(7) == -1


def test_bytes_per_token_and_required_sizes(L):
    cfg = B.make_config(1, 8, 128, 32, max_t=1, max_rows=32768)
    # kb = 8*128/32 = 32 blocks: 32*34 + 32*24 = 1856 bytes per token
    assert B.kvq_bytes_per_token(cfg) == 1856
    sz = B.kvq_required_bytes(cfg)
    # plus one 128-byte column block of padding, rounded up to 256 bytes
    assert sz.k_plane == 32768 * 1088 + 256
    assert sz.v_plane == 32768 * 768 + 256
    assert sz.counters >= (2 * 1 + 1) * 4 and sz.counters % 256 == 0
    assert sz.workspace > 0
    ring = B.make_config(1, 8, 64, 64, max_t=1, window=4096, ring=1)
    sz = B.kvq_required_bytes(ring)
    # ring of window + 31 rows at T = 1
    # planes are padded by one 128-byte column block and rounded up to 256
    # bytes so whole-block tile copies stay inside
    assert sz.k_plane == -(-(4127 * 16 * 34 + 128) // 256) * 256
    assert sz.v_plane == -(-(4127 * 16 * 24 + 128) // 256) * 256
    # FP8 E4M3: one byte per element in both planes
    f8 = B.make_config(1, 8, 128, 32, max_t=1, max_rows=32768, k_fmt=B.KVQ_FP8_E4M3,
                       v_fmt=B.KVQ_FP8_E4M3)
    assert B.kvq_bytes_per_token(f8) == 2 * 1024
    sz = B.kvq_required_bytes(f8)
    assert sz.k_plane == sz.v_plane == 32768 * 1024 + 256


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=48), B.KVQ_EINVAL),           # a block would straddle a head
    (dict(head_dim=0), B.KVQ_EINVAL),
    (dict(max_q_heads=12, n_kv_heads=8), B.KVQ_EINVAL),
    (dict(max_t=0), B.KVQ_EINVAL),
    (dict(max_t=513), B.KVQ_EINVAL),
    (dict(ring=1, window=0), B.KVQ_EINVAL),
    (dict(ring=1, window=100, max_rows=100), B.KVQ_EINVAL),
    (dict(n_seq=0), B.KVQ_EINVAL),
    (dict(max_rows=0), B.KVQ_EINVAL),
])
def test_invalid_configs_rejected(L, kw, status):
    base = dict(n_seq=1, n_kv_heads=2, head_dim=128, max_q_heads=8, max_t=1, max_rows=64,
                window=0, ring=0)
    base.update(kw)
    cfg = B.make_config(**base)
    with pytest.raises(B.KvqError) as e:
        B.kvq_required_bytes(cfg)
    assert e.value.status == status
    # alloc validates before touching the device
    with pytest.raises(B.KvqError) as e:
        B.kvq_alloc(cfg, 16, 16, 16, 16)
    assert e.value.status == status


@pytest.mark.parametrize("k_fmt,v_fmt", [
    (B.KVQ_Q5_1, B.KVQ_Q5_1), (B.KVQ_Q5_1, B.KVQ_Q8_0), (B.KVQ_FP8_E4M3, B.KVQ_Q5_1),
    (B.KVQ_Q8_0, B.KVQ_FP8_E4M3), (9, 9),
])
def test_wrong_formats_unsupported(L, k_fmt, v_fmt):
    cfg = B.make_config(1, 2, 128, 8, max_rows=64, k_fmt=k_fmt, v_fmt=v_fmt)
    with pytest.raises(B.KvqError) as e:
        B.kvq_required_bytes(cfg)
    assert e.value.status == B.KVQ_EUNSUPPORTED


def test_null_and_misaligned_buffers(L):
    cfg = B.make_config(1, 2, 128, 8, max_rows=64)
    with pytest.raises(B.KvqError) as e:
        B.kvq_alloc(cfg, 0, 16, 16, 16)
    assert e.value.status == B.KVQ_EINVAL
    with pytest.raises(B.KvqError) as e:
        B.kvq_alloc(cfg, 16, 17, 16, 16)
    assert e.value.status == B.KVQ_EINVAL
    assert "aligned" in B.kvq_last_error()


def test_null_handle_calls(L):
    for fn, args in [(L.kvq_append, (None, 1, 1, 0, 1, None, 0, None)),
                     (L.kvq_decode, (None, 1, 0, 1, 8, None, 0.0, 1, None)),
                     (L.kvq_truncate, (None, None, None)),
                     (L.kvq_truncate_device, (None, None, 1, None)),
                     (L.kvq_sync_len, (None, None)),
                     (L.kvq_note_replayed, (None, 1, 1))]:
        assert fn(*args) == B.KVQ_EINVAL
