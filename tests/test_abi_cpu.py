"""The C-ABI library without a GPU: it loads, exports every function that
include/*.h declares, and turns each rule of the writer's layout check and
of the call's preconditions into its status code before any CUDA call
(vLLM DSpark context-KV writer page: _validate, __call__,
rotary_dims_supported).  No test here launches a kernel."""

import ctypes
import glob
import os
import re

import pytest

import speculative_decoding_draft_ctx_gb300 as dk
from speculative_decoding_draft_ctx_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return dk.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(dspark_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "dspark_ctx_kv_write" in names and len(names) >= 10
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing
    assert names == set(dk.EXPORTS)


def test_library_is_the_in_tree_build(L):
    assert os.path.dirname(os.path.abspath(L._name)) == os.path.join(ROOT, "speculative_decoding_draft_ctx_gb300")


FAKE = 0x10000  # an aligned address that is never dereferenced: every call below fails validation


def call(**over):
    a = dict(all_kv=FAKE, knorm_w=FAKE, positions=FAKE, slot_mapping=FAKE, num_ctx=4, cos_sin=FAKE,
             max_pos=64, layer0_cache=FAKE, num_blocks=4, cache_offsets=FAKE, k_scales=FAKE,
             v_scales=FAKE, L=2, nkv=2, block_size=16, rotary_dim=32, eps=1e-6, kv_dtype=0)
    a.update(over)
    with pytest.raises(dk.DSparkError) as ei:
        dk.dspark_ctx_kv_write(**a, stream=0)
    return ei.value.name


@pytest.mark.parametrize("r", [0, 8, 48, 96, 128, -16])
def test_unsupported_rotary_dims(L, r):
    assert call(rotary_dim=r) == "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM"


def test_rotary_dims_supported_rule(L):
    for r in (16, 32, 64):
        assert dk.rotary_dims_supported(r, 128)
        assert not dk.rotary_dims_supported(r, 64)
    assert not dk.rotary_dims_supported(128, 128)


@pytest.mark.parametrize("bs", [0, 3, 12, 48, -16])
def test_block_size_must_be_power_of_two(L, bs):
    assert call(block_size=bs) == "DSPARK_ERR_BLOCK_SIZE"


@pytest.mark.parametrize("over", [dict(num_ctx=-1), dict(L=0), dict(nkv=0), dict(num_blocks=0),
                                  dict(max_pos=0), dict(eps=-1.0), dict(eps=float("nan")),
                                  dict(eps=float("inf")), dict(all_kv=0), dict(cos_sin=0),
                                  dict(positions=0), dict(slot_mapping=0), dict(layer0_cache=0),
                                  dict(cache_offsets=0), dict(kv_dtype=1, k_scales=0),
                                  dict(num_ctx=1 << 60)])
def test_invalid_arguments(L, over):
    assert call(**over) == "DSPARK_ERR_INVALID_ARG"


@pytest.mark.parametrize("over", [dict(all_kv=FAKE + 8), dict(knorm_w=FAKE + 2), dict(cos_sin=FAKE + 4),
                                  dict(layer0_cache=FAKE + 8), dict(positions=FAKE + 4),
                                  dict(slot_mapping=FAKE + 1), dict(cache_offsets=FAKE + 4)])
def test_misaligned_buffers(L, over):
    assert call(**over) == "DSPARK_ERR_ALIGNMENT"


@pytest.mark.parametrize("kv", [2, -1, 7])
def test_unknown_kv_dtype(L, kv):
    assert call(kv_dtype=kv) == "DSPARK_ERR_DTYPE"


def test_zero_tokens_is_ok_without_a_device(L):
    dk.dspark_ctx_kv_write(0, 0, 0, 0, 0, 0, 64, 0, 4, 0, 0, 0, 2, 2, 16, 32, 1e-6, 0, stream=0)
    assert dk.dspark_ctx_kv_last_error() == ""


def test_status_strings(L):
    for code, name in dk.STATUS.items():
        assert dk.dspark_ctx_kv_status_string(code) == name


def desc(data=FAKE, shape=(8, 2, 16, 256), stride=None, elem=2, cache_dtype=0, kv=0, scales_ok=1, ndim=4):
    d = dk.CacheDesc()
    d.data = data
    d.ndim = ndim
    if stride is None:
        stride = (shape[1] * shape[2] * shape[3], shape[2] * shape[3], shape[3], 1)
    for i in range(4):
        d.shape[i] = shape[i]
        d.stride[i] = stride[i]
    d.elem_size, d.cache_dtype, d.kv_dtype = elem, cache_dtype, kv
    d.k_scale = d.v_scale = FAKE
    d.scales_ok = scales_ok
    return d


def status_of(descs):
    try:
        dk.dspark_ctx_kv_validate_layers(descs)
        return "DSPARK_OK"
    except dk.DSparkError as e:
        return e.name


def test_layout_rules(L):
    span = 8 * 2 * 16 * 256 * 2
    assert status_of([desc(), desc(data=FAKE + span)]) == "DSPARK_OK"
    assert status_of([desc(elem=1, cache_dtype=1, kv=1), desc(data=FAKE + span, elem=1, cache_dtype=1, kv=1)]) == "DSPARK_OK"
    assert status_of([]) == "DSPARK_ERR_INVALID_ARG"
    assert status_of([desc(data=0)]) == "DSPARK_ERR_INVALID_ARG"  # not bound
    assert status_of([desc(shape=(0, 2, 16, 256))]) == "DSPARK_ERR_INVALID_ARG"
    assert status_of([desc(shape=(8, 2, 16, 128))]) == "DSPARK_ERR_INVALID_ARG"
    assert status_of([desc(ndim=3)]) == "DSPARK_ERR_INVALID_ARG"
    assert status_of([desc(shape=(8, 2, 24, 256))]) == "DSPARK_ERR_BLOCK_SIZE"
    assert status_of([desc(stride=(2 * 16 * 256, 256, 2 * 256, 1))]) == "DSPARK_ERR_INVALID_ARG"
    assert status_of([desc(kv=1)]) == "DSPARK_ERR_DTYPE"  # fp8 cache that is not uint8
    assert status_of([desc(elem=1, cache_dtype=1)]) == "DSPARK_ERR_DTYPE"  # bf16 kv on uint8
    assert status_of([desc(kv=-1)]) == "DSPARK_ERR_DTYPE"
    assert status_of([desc(scales_ok=0)]) == "DSPARK_ERR_INVALID_ARG"
    assert status_of([desc(), desc(data=FAKE + span, shape=(4, 2, 16, 256))]) == "DSPARK_ERR_INVALID_ARG"
    assert status_of([desc(), desc(data=FAKE + span + 16)]) == "DSPARK_ERR_ALIGNMENT"  # 8 elements off
    assert status_of([desc(), desc(data=FAKE - span)]) == "DSPARK_OK"  # negative offset is fine


def test_tables_reject_bad_arguments_without_device(L):
    h = ctypes.c_void_p()
    assert L.dspark_ctx_kv_tables_create(0, ctypes.byref(h)) == dk.STATUS_CODE["DSPARK_ERR_INVALID_ARG"]
    assert L.dspark_ctx_kv_tables_update(None, None, 2, None, None, None) == dk.STATUS_CODE["DSPARK_ERR_INVALID_ARG"]
    assert L.dspark_ctx_kv_tables_builds(None) == 0
    L.dspark_ctx_kv_tables_destroy(None)


# ------------------------------------------------------------ draft-token QK insert
# (DSpark draft model page, dspark_qknorm_rope_kv_insert; layout and fp8 rules
# of the context-KV writer page)

def qk_call(expect_ok=False, **over):
    a = dict(qkv=FAKE, q_norm_w=FAKE, k_norm_w=FAKE, cos_sin=FAKE, max_pos=64, positions=FAKE, num_tokens=7,
             num_heads=4, num_kv_heads=1, rotary_dim=64, eps=1e-6, slot_mapping=FAKE, kv_cache=FAKE,
             num_blocks=4, block_size=16, kv_dtype=0, k_scale=None, v_scale=None, q_fp8_out=None,
             q_fp8_scale=1.0)
    a.update(over)
    if expect_ok:
        dk.dspark_qknorm_rope_kv_insert(**a, stream=0)
        return "DSPARK_OK"
    with pytest.raises(dk.DSparkError) as ei:
        dk.dspark_qknorm_rope_kv_insert(**a, stream=0)
    return ei.value.name


def test_qk_insert_argument_checks(L):
    assert qk_call(rotary_dim=48) == "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM"
    assert qk_call(num_tokens=-1) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(num_heads=0) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(num_kv_heads=0) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(max_pos=0) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(eps=float("nan")) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(eps=-1.0) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(block_size=24) == "DSPARK_ERR_BLOCK_SIZE"
    assert qk_call(kv_dtype=7) == "DSPARK_ERR_DTYPE"
    assert qk_call(num_blocks=0) == "DSPARK_ERR_INVALID_ARG"
    # the insert needs both a slot mapping and a cache
    assert qk_call(kv_cache=None) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(slot_mapping=None) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(q_fp8_out=FAKE, q_fp8_scale=0.0) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(q_fp8_out=FAKE, q_fp8_scale=float("inf")) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(qkv=None) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(positions=None) == "DSPARK_ERR_INVALID_ARG"
    assert qk_call(qkv=FAKE + 8) == "DSPARK_ERR_ALIGNMENT"
    assert qk_call(kv_cache=FAKE + 8) == "DSPARK_ERR_ALIGNMENT"
    assert qk_call(q_fp8_out=FAKE + 8) == "DSPARK_ERR_ALIGNMENT"
    assert qk_call(positions=FAKE + 4) == "DSPARK_ERR_ALIGNMENT"
    assert qk_call(error_flags=FAKE + 2) == "DSPARK_ERR_ALIGNMENT"
    # without an insert the cache arguments are not looked at
    assert qk_call(slot_mapping=None, kv_cache=None, block_size=24, kv_dtype=7, num_tokens=0,
                   expect_ok=True) == "DSPARK_OK"
    # no tokens: OK without a launch
    assert qk_call(num_tokens=0, expect_ok=True) == "DSPARK_OK"
    assert qk_call(rotary_dim=48) == "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM"
    assert "not in {16, 32, 64}" in dk.dspark_ctx_kv_last_error()


def test_norm_argument_checks(L):
    def norm(**over):
        a = dict(x=FAKE, w=FAKE, out=FAKE, rows=4, hidden=4096, eps=1e-6)
        a.update(over)
        with pytest.raises(dk.DSparkError) as ei:
            dk.dspark_gemma_rms_norm(**a, stream=0)
        return ei.value.name
    assert norm(hidden=100) == "DSPARK_ERR_INVALID_ARG"
    assert norm(hidden=8200) == "DSPARK_ERR_INVALID_ARG"
    assert norm(rows=-1) == "DSPARK_ERR_INVALID_ARG"
    assert norm(eps=float("inf")) == "DSPARK_ERR_INVALID_ARG"
    assert norm(x=None) == "DSPARK_ERR_INVALID_ARG"
    assert norm(x=FAKE + 8) == "DSPARK_ERR_ALIGNMENT"
    assert norm(out=FAKE + 16) == "DSPARK_ERR_INVALID_ARG"  # overlaps x without being x
    dk.dspark_gemma_rms_norm(FAKE, FAKE, FAKE, 0, 4096, 1e-6, stream=0)  # no rows: no launch


def test_projection_argument_checks(L):
    def proj(**over):
        a = dict(x=FAKE, w_kv=FAKE, all_kv_out=FAKE, num_ctx=4, hidden=4096, L=2, nkv=2)
        a.update(over)
        with pytest.raises(dk.DSparkError) as ei:
            dk.dspark_ctx_kv_project(**a, stream=0)
        return ei.value.name
    assert proj(hidden=100) == "DSPARK_ERR_ALIGNMENT"
    assert proj(L=0) == "DSPARK_ERR_INVALID_ARG"
    assert proj(nkv=40000) == "DSPARK_ERR_INVALID_ARG"
    assert proj(num_ctx=-1) == "DSPARK_ERR_INVALID_ARG"
    assert proj(num_ctx=65535 * 128 + 1) == "DSPARK_ERR_INVALID_ARG"
    assert proj(x=FAKE + 8) == "DSPARK_ERR_ALIGNMENT"
    assert proj(all_kv_out=None) == "DSPARK_ERR_ALIGNMENT"
    dk.dspark_ctx_kv_project(FAKE, FAKE, FAKE, 0, 4096, 2, 2, stream=0)  # no tokens: no launch
    with pytest.raises(dk.DSparkError) as ei:
        dk.dspark_ctx_kv_project_write(FAKE, FAKE, 4, 4096, FAKE, FAKE, FAKE, FAKE, 64, FAKE, 4, FAKE, FAKE, FAKE,
                                       33, 1, 16, 32, 1e-6, 0, stream=0)
    assert ei.value.name == "DSPARK_ERR_INVALID_ARG"  # more than 32 layers
    with pytest.raises(dk.DSparkError) as ei:
        dk.dspark_ctx_kv_project_write(FAKE, FAKE, 4, 4096, FAKE, FAKE, FAKE, FAKE, 64, FAKE, 4, FAKE, FAKE, FAKE,
                                       2, 1, 16, 48, 1e-6, 0, stream=0)
    assert ei.value.name == "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM"


# ------------------------------------------------------------ the general write
# (layouts the writer page's _validate / rotary_dims_supported refuse)

def gcall(expect_ok=False, **over):
    a = dict(all_kv=FAKE, knorm_w=FAKE, positions=FAKE, slot_mapping=FAKE, layer_slot_mappings=None, num_ctx=4,
             cos_sin=FAKE, max_pos=64, layer0_cache=FAKE, num_blocks=4, cache_offsets=FAKE, k_scales=FAKE,
             v_scales=FAKE, L=2, nkv=2, head_dim=64, block_size=24, rotary_dim=18, eps=1e-6, kv_dtype=0)
    a.update(over)
    if expect_ok:
        dk.dspark_ctx_kv_write_general(**a, stream=0)
        return "DSPARK_OK"
    with pytest.raises(dk.DSparkError) as ei:
        dk.dspark_ctx_kv_write_general(**a, stream=0)
    return ei.value.name


def test_general_write_argument_checks(L):
    for hd in (0, 32, 96, 192, 512):
        assert gcall(head_dim=hd) == "DSPARK_ERR_INVALID_ARG"
    for hd, r in ((64, 0), (64, 7), (64, 66), (128, 130), (256, 258), (256, -2)):
        assert gcall(head_dim=hd, rotary_dim=r) == "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM"
    for bs in (0, -3):
        assert gcall(block_size=bs) == "DSPARK_ERR_BLOCK_SIZE"
    # exactly one slot source
    assert gcall(layer_slot_mappings=FAKE) == "DSPARK_ERR_INVALID_ARG"
    assert gcall(slot_mapping=None) == "DSPARK_ERR_INVALID_ARG"
    assert gcall(slot_mapping=None, layer_slot_mappings=FAKE + 4) == "DSPARK_ERR_ALIGNMENT"
    assert gcall(kv_dtype=3) == "DSPARK_ERR_DTYPE"
    assert gcall(eps=float("nan")) == "DSPARK_ERR_INVALID_ARG"
    assert gcall(num_blocks=1 << 58) == "DSPARK_ERR_INVALID_ARG"
    for over in (dict(all_kv=FAKE + 8), dict(knorm_w=FAKE + 8), dict(cos_sin=FAKE + 4),
                 dict(layer0_cache=FAKE + 8), dict(cache_offsets=FAKE + 4), dict(error_flags=FAKE + 2)):
        assert gcall(**over) == "DSPARK_ERR_ALIGNMENT"
    # the pages' layout through the general entry: the same buffer checks
    assert gcall(head_dim=128, rotary_dim=32, block_size=16, all_kv=FAKE + 8) == "DSPARK_ERR_ALIGNMENT"
    # no tokens: OK, no launch, no slot source needed
    assert gcall(num_ctx=0, slot_mapping=None, expect_ok=True) == "DSPARK_OK"


def test_sched_write_argument_checks(L):
    """dspark_ctx_kv_write_sched: exactly one slot source, an 8-byte aligned
    work counter and pointer table, the write's own checks -- all before any
    CUDA call."""
    def scall(expect_ok=False, **over):
        a = dict(all_kv=FAKE, knorm_w=FAKE, positions=FAKE, slot_mapping=FAKE, layer_slot_mappings=None, num_ctx=4,
                 cos_sin=FAKE, max_pos=64, layer0_cache=FAKE, num_blocks=4, cache_offsets=FAKE, k_scales=FAKE,
                 v_scales=FAKE, L=2, nkv=2, block_size=16, rotary_dim=32, eps=1e-6, kv_dtype=0, error_flags=None,
                 work_counter=None)
        a.update(over)
        if expect_ok:
            dk.dspark_ctx_kv_write_sched(**a, stream=0)
            return "DSPARK_OK"
        with pytest.raises(dk.DSparkError) as ei:
            dk.dspark_ctx_kv_write_sched(**a, stream=0)
        return ei.value.name

    assert scall(slot_mapping=None) == "DSPARK_ERR_INVALID_ARG"                      # no slot source
    assert scall(layer_slot_mappings=FAKE) == "DSPARK_ERR_INVALID_ARG"               # two
    assert scall(slot_mapping=None, layer_slot_mappings=FAKE + 4) == "DSPARK_ERR_ALIGNMENT"
    assert scall(work_counter=FAKE + 4) == "DSPARK_ERR_ALIGNMENT"                     # counter: 8-byte words
    assert scall(rotary_dim=24) == "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM"
    assert scall(block_size=48) == "DSPARK_ERR_BLOCK_SIZE"
    assert scall(num_ctx=0, slot_mapping=None, expect_ok=True) == "DSPARK_OK"       # nothing to store


def test_no_alloc_write_argument_checks(L):
    """dspark_ctx_kv_write_noalloc refuses a layer count beyond its fixed
    device array, and its host-table rules, before any CUDA call."""
    def ncall(expect_ok=False, **over):
        a = dict(all_kv=FAKE, knorm_w=FAKE, positions=FAKE, slot_mapping=FAKE, layer_slot_mappings=None, num_ctx=4,
                 cos_sin=FAKE, max_pos=64, layer0_cache=FAKE, num_blocks=4, cache_offsets=[0, 4096],
                 k_scales=[FAKE, FAKE], v_scales=[FAKE, FAKE], L=2, nkv=2, block_size=16, rotary_dim=32,
                 eps=1e-6, kv_dtype=0)
        a.update(over)
        if expect_ok:
            dk.dspark_ctx_kv_write_noalloc(**a, stream=0)
            return "DSPARK_OK"
        with pytest.raises(dk.DSparkError) as ei:
            dk.dspark_ctx_kv_write_noalloc(**a, stream=0)
        return ei.value.name, str(ei.value)

    name, msg = ncall(L=65, cache_offsets=[0] * 65, k_scales=[FAKE] * 65, v_scales=[FAKE] * 65)
    assert name == "DSPARK_ERR_INVALID_ARG" and "1 to 64 layers" in msg
    assert ncall(L=0, cache_offsets=[0], k_scales=None, v_scales=None)[0] == "DSPARK_ERR_INVALID_ARG"
    assert ncall(slot_mapping=None)[0] == "DSPARK_ERR_INVALID_ARG"  # no slot source
    assert ncall(layer_slot_mappings=[FAKE, FAKE])[0] == "DSPARK_ERR_INVALID_ARG"  # two
    assert ncall(slot_mapping=None, layer_slot_mappings=[FAKE, None])[0] == "DSPARK_ERR_INVALID_ARG"
    assert ncall(kv_dtype=1, k_scales=None)[0] == "DSPARK_ERR_INVALID_ARG"  # fp8 needs scales
    assert ncall(cache_offsets=[0, 4100])[0] == "DSPARK_ERR_ALIGNMENT"  # not 16 elements apart
    assert ncall(num_ctx=-1)[0] == "DSPARK_ERR_INVALID_ARG"
    assert ncall(num_ctx=0, expect_ok=True) == "DSPARK_OK"  # nothing to store, no CUDA call


def test_general_supported_rule(L):
    for hd in (64, 128, 256):
        for r in range(2, hd + 1, 2):
            assert dk.general_layout_supported(hd, r, 1)
        assert not dk.general_layout_supported(hd, hd + 2, 16)
        assert not dk.general_layout_supported(hd, 3, 16)
        assert not dk.general_layout_supported(hd, 16, 0)
    assert dk.general_layout_supported(128, 32, 48)
    assert not dk.general_layout_supported(96, 32, 16)


def test_general_layout_rules(L):
    def general_status(descs):
        try:
            dk.dspark_ctx_kv_validate_layers_general(descs)
            return "DSPARK_OK"
        except dk.DSparkError as e:
            return e.name

    for last in (128, 256, 512):
        assert general_status([desc(shape=(8, 2, 24, last))]) == "DSPARK_OK"
    assert general_status([desc(shape=(8, 2, 24, 384))]) == "DSPARK_ERR_INVALID_ARG"
    assert general_status([desc(shape=(8, 2, 1, 128))]) == "DSPARK_OK"
    assert status_of([desc(shape=(8, 2, 24, 256))]) == "DSPARK_ERR_BLOCK_SIZE"  # the pages' rule
    assert status_of([desc(shape=(8, 2, 16, 512))]) == "DSPARK_ERR_INVALID_ARG"
    span = 8 * 2 * 24 * 512 * 2
    assert general_status([desc(shape=(8, 2, 24, 512)), desc(data=FAKE + span + 16, shape=(8, 2, 24, 512))]) == \
        "DSPARK_ERR_ALIGNMENT"


# ---------------------------------------------------------------- tensor checks of the Python API
# The library receives only addresses, so the Python layer checks every
# tensor's dtype, device, contiguity and extent before the call (the pages'
# writer validates its inputs before the launch).  A writer object is built
# here around CPU caches without its device tables; reaching the library is
# replaced by a sentinel, so no test here touches a GPU.

class _Reached(Exception):
    pass


def _stop(*a, **k):
    raise _Reached()


def _cpu_writer(monkeypatch, L=2, H=2, bs=16, nb=4):
    import torch
    from speculative_decoding_draft_ctx_gb300 import writer as wr

    w = object.__new__(wr.ContextKVWriter)
    w.kv_caches = [torch.empty(nb, H, bs, 256, dtype=torch.bfloat16) for _ in range(L)]
    w.k_scales = w.v_scales = [torch.ones(1) for _ in range(L)]
    w.kv_cache_dtype, w.general, w._dtype, w._flags = "auto", False, 0, None
    w.num_layers, w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim = L, nb, H, bs, 128
    monkeypatch.setattr(w, "ensure_tables", _stop)
    monkeypatch.setattr(wr, "dspark_ctx_kv_project_write", _stop)
    return w


def _good_write_args(T=4, L=2, H=2, r=32):
    import torch

    bf = torch.bfloat16
    return dict(all_kv=torch.zeros(T, L, 2, H, 128, dtype=bf), k_norm_weight=torch.zeros(L, 128, dtype=bf),
                eps=1e-6, positions=torch.zeros(T, dtype=torch.int64), cos_sin_cache=torch.zeros(64, r, dtype=bf),
                rotary_dim=r, slot_mapping=torch.zeros(T, dtype=torch.int64))


def _bad_write_cases():
    import torch

    bf = torch.bfloat16
    return [
        ("positions", torch.zeros(4, dtype=torch.int32)),           # read as int64: 8T bytes from 4T
        ("slot_mapping", torch.zeros(4, dtype=torch.int32)),
        ("positions", torch.zeros(3, dtype=torch.int64)),           # fewer entries than tokens
        ("slot_mapping", torch.zeros(3, dtype=torch.int64)),
        ("positions", torch.zeros(8, dtype=torch.int64)[::2]),      # not contiguous
        ("cos_sin_cache", torch.zeros(64, 16, dtype=bf)),          # narrower than rotary_dim
        ("cos_sin_cache", torch.zeros(64, 32, dtype=torch.float32)),
        ("cos_sin_cache", torch.zeros(64, 64, dtype=bf)[:, :32]),  # right width, not contiguous
        ("k_norm_weight", torch.zeros(128, dtype=bf)),             # [128], not [L, 128]
        ("k_norm_weight", torch.zeros(2, 128, dtype=torch.float32)),
        ("all_kv", torch.zeros(4, 2, 2, 2, 256, dtype=bf)[..., :128]),
        ("all_kv", torch.zeros(4, 2, 2, 2, 128, dtype=torch.float32)),
        ("all_kv", torch.zeros(4, 2, 2, 2, 128, dtype=bf, device="meta")),  # not on the caches' device
        ("positions", torch.zeros(4, dtype=torch.int64, device="meta")),
        ("error_flags", torch.zeros(1, dtype=torch.int64)),
        ("error_flags", torch.zeros(0, dtype=torch.int32)),
    ]


def test_writer_passes_good_tensors_to_the_library(monkeypatch):
    w = _cpu_writer(monkeypatch)
    with pytest.raises(_Reached):
        w(**_good_write_args())
    import torch

    a = _good_write_args()
    a["slot_mapping"] = [torch.zeros(4, dtype=torch.int64), torch.ones(4, dtype=torch.int64)]
    with pytest.raises(_Reached):
        w(**a)


@pytest.mark.parametrize("case", range(16))
def test_writer_refuses_bad_tensors(monkeypatch, case):
    name, bad = _bad_write_cases()[case]
    w = _cpu_writer(monkeypatch)
    a = _good_write_args()
    a[name] = bad
    with pytest.raises(dk.DSparkError) as ei:
        w(**a)
    assert ei.value.name == "DSPARK_ERR_INVALID_ARG"


def test_writer_work_counters_per_stream_and_never_made_under_capture(monkeypatch):
    """The dynamic tail's counters: one per stream, made zeroed (and waited
    for) at the first call there outside capture and reused after; a call
    captured on a stream without one gets none (the fixed split) and makes
    none, and an existing counter serves captured calls on its stream."""
    import torch
    from speculative_decoding_draft_ctx_gb300 import writer as wr

    w = _cpu_writer(monkeypatch)
    w._work = {}
    capturing = [False]
    syncs = []

    class FakeStream:
        def __init__(self, h):
            self.cuda_stream = h

        def synchronize(self):
            syncs.append(self.cuda_stream)

    cur = FakeStream(7)
    monkeypatch.setattr(torch.cuda, "is_current_stream_capturing", lambda: capturing[0])
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: cur)
    monkeypatch.setattr(wr, "_stream_handle", lambda s: cur.cuda_stream if s is None else s)
    c7 = w._work_counter(None)
    assert c7.dtype == torch.int64 and c7.tolist() == [0, 0] and syncs == [7]
    assert w._work_counter(None) is c7 and syncs == [7]  # reused, no second wait
    c11 = w._work_counter(11)
    assert c11 is not c7 and c11.tolist() == [0, 0]
    capturing[0] = True
    assert w._work_counter(13) is None and 13 not in w._work
    assert w._work_counter(11) is c11
    assert len(syncs) == 2


def test_writer_refuses_bad_per_layer_slot_mapping(monkeypatch):
    import torch

    w = _cpu_writer(monkeypatch)
    a = _good_write_args()
    a["slot_mapping"] = [torch.zeros(4, dtype=torch.int64), torch.zeros(4, dtype=torch.int32)]
    with pytest.raises(dk.DSparkError, match="slot_mapping\\[1\\]"):
        w(**a)


def test_project_and_write_refuses_bad_tensors(monkeypatch):
    import torch

    bf = torch.bfloat16
    w = _cpu_writer(monkeypatch)
    a = _good_write_args()
    good = dict(context_states=torch.zeros(4, 64, dtype=bf), w_kv=torch.zeros(2 * 2 * 2 * 128, 64, dtype=bf),
                k_norm_weight=a["k_norm_weight"], eps=1e-6, positions=a["positions"],
                cos_sin_cache=a["cos_sin_cache"], rotary_dim=32, slot_mapping=a["slot_mapping"])
    with pytest.raises(_Reached):
        w.project_and_write(**good)
    for name, bad in [("context_states", torch.zeros(4, 64)), ("context_states", torch.zeros(4, 128, dtype=bf)[:, ::2]),
                      ("w_kv", torch.zeros(1024, 64)), ("positions", torch.zeros(4, dtype=torch.int32)),
                      ("slot_mapping", torch.zeros(2, dtype=torch.int64)),
                      ("cos_sin_cache", torch.zeros(64, 16, dtype=bf)), ("k_norm_weight", torch.zeros(128, dtype=bf))]:
        b = dict(good)
        b[name] = bad
        with pytest.raises(dk.DSparkError) as ei:
            w.project_and_write(**b)
        assert ei.value.name == "DSPARK_ERR_INVALID_ARG", name


def test_qk_insert_refuses_bad_tensors(monkeypatch):
    import torch
    from speculative_decoding_draft_ctx_gb300 import writer as wr

    monkeypatch.setattr(wr, "dspark_qknorm_rope_kv_insert", _stop)
    bf = torch.bfloat16
    T, Hq, Hkv = 3, 4, 1
    good = dict(qkv=torch.zeros(T, (Hq + 2 * Hkv) * 128, dtype=bf), q_norm_weight=torch.zeros(128, dtype=bf),
                k_norm_weight=torch.zeros(128, dtype=bf), cos_sin_cache=torch.zeros(64, 64, dtype=bf),
                positions=torch.zeros(T, dtype=torch.int64), num_heads=Hq, num_kv_heads=Hkv, rotary_dim=64,
                eps=1e-6, slot_mapping=torch.zeros(T, dtype=torch.int64),
                kv_cache=torch.zeros(4, Hkv, 16, 256, dtype=torch.uint8), k_scale=torch.ones(1),
                v_scale=torch.ones(1), q_fp8_out=torch.zeros(T, Hq * 128, dtype=torch.uint8))
    with pytest.raises(_Reached):
        wr.qknorm_rope_kv_insert(**good)
    for name, bad in [("qkv", torch.zeros(T, (Hq + 2 * Hkv) * 128)), ("q_norm_weight", torch.zeros(2, 128, dtype=bf)),
                      ("k_norm_weight", torch.zeros(128)), ("cos_sin_cache", torch.zeros(64, 32, dtype=bf)),
                      ("positions", torch.zeros(T, dtype=torch.int32)), ("slot_mapping", torch.zeros(2, dtype=torch.int64)),
                      ("kv_cache", torch.zeros(4, Hkv, 16, 256, dtype=torch.float16)),
                      ("kv_cache", torch.zeros(4, Hkv, 16, 512, dtype=torch.uint8)[..., :256]),
                      ("k_scale", torch.ones(1, dtype=torch.float64)), ("v_scale", torch.ones(0)),
                      ("q_fp8_out", torch.zeros(T, Hq * 128 - 1, dtype=torch.uint8)),
                      ("qkv", torch.zeros(T, (Hq + 2 * Hkv) * 128, dtype=bf, device="meta"))]:
        b = dict(good)
        b[name] = bad
        with pytest.raises(dk.DSparkError) as ei:
            wr.qknorm_rope_kv_insert(**b)
        assert ei.value.name == "DSPARK_ERR_INVALID_ARG", name


def test_projection_and_norm_refuse_bad_tensors(monkeypatch):
    import torch
    from speculative_decoding_draft_ctx_gb300 import writer as wr

    monkeypatch.setattr(wr, "dspark_ctx_kv_project", _stop)
    monkeypatch.setattr(wr, "dspark_gemma_rms_norm", _stop)
    bf = torch.bfloat16
    x, w = torch.zeros(4, 64, dtype=bf), torch.zeros(2 * 2 * 2 * 128, 64, dtype=bf)
    with pytest.raises(_Reached):
        wr.project_context_kv(x, w, 2, 2)
    for args in [(torch.zeros(4, 64), w), (x, torch.zeros(1024, 32, dtype=bf)), (x, w.t().contiguous())]:
        with pytest.raises(dk.DSparkError):
            wr.project_context_kv(*args, 2, 2)
    with pytest.raises(dk.DSparkError):
        wr.project_context_kv(x, w, 2, 2, out=torch.zeros(4, 1000, dtype=bf))
    with pytest.raises(_Reached):
        wr.gemma_rms_norm(x, torch.zeros(64, dtype=bf), 1e-6)
    for args in [(torch.zeros(4, 64), torch.zeros(64, dtype=bf)), (x, torch.zeros(32, dtype=bf)),
                 (x, torch.zeros(64))]:
        with pytest.raises(dk.DSparkError):
            wr.gemma_rms_norm(*args, 1e-6)
    with pytest.raises(dk.DSparkError):
        wr.gemma_rms_norm(x, torch.zeros(64, dtype=bf), 1e-6, out=torch.zeros(4, 32, dtype=bf))
