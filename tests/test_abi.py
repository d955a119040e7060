"""The C-ABI library builds, loads without a GPU, exports every declared entry point,
and answers the host-only queries (no kernel is launched here)."""
import ctypes as C
import os
import re

import pytest

from oracle import Oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_lora.h")


@pytest.fixture(scope="module")
def ml():
    from expert_gemm_gb300 import build, moe_lora
    build.build()
    moe_lora.load()
    return moe_lora


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_lora_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(ml):
    lib = C.CDLL(ml.LIB_PATH)
    syms = declared_symbols()
    assert len(syms) >= 11
    for s in syms:
        assert hasattr(lib, s), s
    assert sorted(ml.EXPORTS) == syms


def test_version_and_status_strings(ml):
    lib = ml.load()
    assert lib.moe_lora_version() >= 100
    for st in range(7):
        assert lib.moe_lora_status_string(st)


def _dims(ml, **kw):
    base = dict(T=64, H=256, I=512, E=8, k=2, L=4, r_max=8, block_m=16, ranks=(8, 8, 8, 8))
    base.update(kw)
    return ml.LayerDims(**base)


def test_capacity_matches_oracle_bound(ml):
    for T, k, E, L, BM in [(64, 2, 8, 4, 16), (16, 4, 32, 8, 16), (25600, 4, 32, 8, 128), (4096, 8, 128, 64, 64),
                           (1, 8, 128, 64, 16), (0, 2, 8, 4, 16)]:
        d = _dims(ml, T=T, k=k, E=E, L=L, block_m=BM, r_max=16, ranks=(16,) * L)
        assert ml.align_capacity(d) == Oracle.capacity(T, E, k, L, BM)


def test_host_validation(ml):
    bad = [dict(H=100), dict(I=0), dict(E=0), dict(k=9), dict(block_m=24), dict(r_max=12),
           dict(ranks=(8, 0, 8, 8)), dict(ranks=(8, 16, 8, 8)), dict(L=300, ranks=(8,) * 300), dict(T=-1)]
    for kw in bad:
        with pytest.raises(ml.MoeLoraError) as ei:
            ml.workspace_size(_dims(ml, **kw))
        assert ei.value.status in (ml.EINVAL, ml.EUNSUPPORTED), kw
    a, f = ml.workspace_size(_dims(ml))
    assert a > 0 and f > 0
    assert ml.layer_workspace_size(_dims(ml)) > a + f


def test_pick_block_m(ml):
    assert ml.pick_block_m(16, 4, 32) == 16
    assert ml.pick_block_m(25600, 4, 32) == 256
    assert ml.pick_block_m(256, 8, 128) in (16, 32)
    assert ml.pick_block_m(4096, 8, 128) == 128


def test_null_and_misaligned_pointers_rejected_before_launch(ml):
    """Invalid pointers are refused on the host; nothing reaches a device."""
    lib = ml.load()
    d = _dims(ml)
    dc = d.c()
    bufs = ml.AlignBuf(16, 16, 16, 16, 16, 16)
    st = lib.moe_lora_forward(C.byref(dc), None, None, C.byref(bufs), None, None, None, None, None, None, None,
                              None, 0, 16, None, None)
    assert st == ml.EINVAL
    st = lib.moe_lora_forward(C.byref(dc), 18, 16, C.byref(bufs), 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, 16,
                              None, None)
    assert st == ml.EALIGN
    st = lib.moe_lora_forward(C.byref(dc), 16, 16, C.byref(bufs), 16, 16, 16, 16, 16, 16, 16, 16, 8, 16,
                              None, None)
    assert st == ml.EWORKSPACE
    st = lib.moe_lora_route(None, 4, 8, 9, None, None, None)
    assert st == ml.EINVAL
