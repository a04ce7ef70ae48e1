"""The C ABI without a GPU: the library builds, loads, exports every declared symbol, and
rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import workload as wl
from shared_kv_concurrent_gb300 import binding, config_for
from shared_kv_concurrent_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "hogwild.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return sorted(set(re.findall(r"\b(hw_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "hw_concurrent_attention" in names and "hw_append_kv" in names and "hw_step_end" in names
    raw = ctypes.CDLL(binding.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert sorted(binding.EXPORTED) == names


def test_status_strings(lib):
    assert binding.hw_status_string(binding.HW_OK) == "HW_OK"
    assert binding.hw_status_string(binding.HW_ERR_OUT_OF_PAGES) == "HW_ERR_OUT_OF_PAGES"
    assert binding.hw_status_string(99) == "HW_ERR_UNKNOWN"


def _cfg(w):
    return config_for(num_problems=w.num_problems, num_workers=w.num_workers,
                      num_layers=w.num_layers, num_q_heads=w.num_q_heads,
                      num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=w.page_size,
                      num_pages=w.num_pages(), max_position=w.max_position(),
                      rope_theta=w.rope_theta, contiguous=w.contiguous)


@pytest.mark.parametrize("name", sorted(wl.CONFIGS))
def test_sizes(lib, name):
    w = wl.CONFIGS[name]()
    cfg = _cfg(w)
    pool = binding.hw_pool_size(cfg)
    assert pool == w.num_layers * w.num_pages() * w.num_kv_heads * w.page_size * w.head_dim * 2
    ws = binding.hw_workspace_size(cfg)
    rope_table = 2 * w.max_position() * w.head_dim // 2 * 4
    assert rope_table < ws < rope_table + (1 << 31)


@pytest.mark.parametrize("field,value", [("head_dim", 96), ("page_size", 100), ("page_size", 0),
                                         ("num_q_heads", 12), ("num_workers", 0),
                                         ("num_workers", 17), ("rope_theta", 0.5),
                                         ("contiguous", 2), ("num_pages", 0), ("layout", 4),
                                         ("layout", -1), ("reserved", 1)])
def test_invalid_config_rejected(lib, field, value):
    cfg = _cfg(wl.tiny())
    cfg.num_q_heads, cfg.num_kv_heads = 64, 8
    setattr(cfg, field, value)
    with pytest.raises(binding.HogwildError) as e:
        binding.hw_workspace_size(cfg)
    assert e.value.status == binding.HW_ERR_INVALID_ARG


@pytest.mark.parametrize("layout", ["combined", "step_wise", "contiguous", "no_sync"])
def test_every_layout_accepted(lib, layout):
    w = wl.tiny()
    cfg = config_for(num_problems=1, num_workers=2, num_layers=1, num_q_heads=8, num_kv_heads=2,
                     head_dim=64, page_size=256, num_pages=8, max_position=1024,
                     rope_theta=1e4, layout=layout)
    assert binding.hw_workspace_size(cfg) > 0 and w.layout == "combined"


def test_null_arguments_rejected_before_cuda(lib):
    cfg = _cfg(wl.tiny())
    ctx = ctypes.c_void_p()
    st = lib.hw_create(ctypes.byref(cfg), None, None, None, 0, None, None, ctypes.byref(ctx))
    assert st == binding.HW_ERR_INVALID_ARG and not ctx.value
    n = (ctypes.c_int32 * 3)(0, 1, 1)
    assert lib.hw_append_kv(None, 0, n, None, None, None) == binding.HW_ERR_INVALID_ARG
    assert lib.hw_concurrent_attention(None, 0, None, None, 0, None, None) == binding.HW_ERR_INVALID_ARG
    assert lib.hw_step_end(None, None, None) == binding.HW_ERR_INVALID_ARG
    a, b = ctypes.c_int32(), ctypes.c_int32()
    assert lib.hw_get_counts(None, ctypes.byref(a), ctypes.byref(b)) == binding.HW_ERR_INVALID_ARG
    assert lib.hw_debug_expire_plans(None, 1) == binding.HW_ERR_INVALID_ARG
    nq = (ctypes.c_int32 * 2)(1, 1)
    assert lib.hw_concurrent_attention_mq(None, 0, None, nq, None, 0, None, None) == \
        binding.HW_ERR_INVALID_ARG
    rg = (ctypes.c_int64 * 2)(0, 1)
    assert lib.hw_concurrent_attention_range(None, 0, None, rg, None, None, None) == \
        binding.HW_ERR_INVALID_ARG
    assert lib.hw_concurrent_attention_noalloc(None, 0, None, None, 0, None, None) == \
        binding.HW_ERR_INVALID_ARG
    assert lib.hw_compact_segments(None, 0, 0, 2, None) == binding.HW_ERR_INVALID_ARG
    merged = ctypes.c_int32()
    assert lib.hw_compact_auto(None, 2, None, ctypes.byref(merged)) == binding.HW_ERR_INVALID_ARG
    size = ctypes.c_size_t()
    assert lib.hw_step_scratch_size(None, n, 0, ctypes.byref(size)) == binding.HW_ERR_INVALID_ARG
    assert lib.hw_decode_step_host(None, n, None, 0, None, 0, None, None, 0, 1, None) == \
        binding.HW_ERR_INVALID_ARG
    # the merge needs no context: bad shapes are refused before any CUDA call
    assert lib.hw_merge_attention(0, 4, 128, None, None, None, 0, None, None) == \
        binding.HW_ERR_INVALID_ARG
    assert lib.hw_merge_attention(2, 4, 6, None, None, None, 0, None, None) == \
        binding.HW_ERR_INVALID_ARG
    lib.hw_destroy(None)


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "shared_kv_concurrent_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                with open(os.path.join(dirpath, f)) as fh:
                    txt = fh.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, re.M), f
