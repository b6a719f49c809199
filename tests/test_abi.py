"""The C-ABI library loads and exports every entry point include/qmoe.h declares.

CPU only: no call here launches GPU work.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qmoe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_mixture_experts_f32_gb300 as q
    return q


def test_every_declared_symbol_is_exported(q):
    names = _declared()
    assert "qmoe_forward" in names and "qmoe_create" in names
    lib = ctypes.CDLL(q.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(q.EXPORTED) == names


def test_expert_stride_matches_page_sizes(q):
    assert q.qmoe_expert_stride(q.QMOE_Q4_K, 768, 2048) == 884736
    assert q.qmoe_expert_stride(q.QMOE_Q6_K, 2048, 768) == 1290240
    assert q.qmoe_expert_stride(q.QMOE_Q4_K, 2048, 768) == 884736
    assert q.qmoe_expert_stride(q.QMOE_Q4_K, 768, 2000) == 0
    assert q.qmoe_expert_stride(7, 768, 2048) == 0


def test_workspace_bytes_and_bad_configs(q):
    ok = q.make_config(2048, 128, 8, 768, 512)
    assert q.qmoe_workspace_bytes(ok) > 512 * 8 * (768 + 2048) * 4
    for bad in (q.make_config(2000, 128, 8, 768, 1), q.make_config(2048, 128, 0, 768, 1),
                q.make_config(2048, 4, 8, 768, 1), q.make_config(2048, 128, 8, 700, 1),
                q.make_config(2048, 128, 8, 768, 0),
                q.make_config(2048, 128, 8, 768, 1, n_heads=32, n_kv_heads=3, head_dim=128,
                              max_ctx=16, rope_base=1e7, rms_eps=1e-6)):
        assert q.qmoe_workspace_bytes(bad) == 0


def test_max_ctx_bound(q):
    # the split-K attention merge keeps two floats per 64 positions in shared
    # memory: contexts up to 2^18 positions are served, longer ones refused
    geo = dict(n_heads=32, n_kv_heads=4, head_dim=128, rope_base=1e7, rms_eps=1e-6)
    assert q.qmoe_workspace_bytes(q.make_config(2048, 128, 8, 768, 1, max_ctx=1 << 18, **geo)) > 0
    assert q.qmoe_workspace_bytes(q.make_config(2048, 128, 8, 768, 1, max_ctx=(1 << 18) + 1, **geo)) == 0


def test_create_rejects_bad_config_before_touching_cuda(q):
    with pytest.raises(q.QmoeError) as ei:
        q.qmoe_create(q.make_config(2048, 128, 17, 768, 1))
    assert ei.value.status == 1
    assert "top_k=17" in q.qmoe_last_error(None) and "top_k=17" in str(ei.value)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "quantized_mixture_experts_f32_gb300")
    for dp, _, fs in os.walk(pkg):
        for f in fs:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dp, f)).read()
                assert not re.search(r"(import\s+oracle|from\s+oracle|qmoe_oracle)", txt), f
