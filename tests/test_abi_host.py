"""Host-side checks of the C ABI: the library loads, exports every declared symbol, and
rejects bad arguments with a status code before touching a GPU."""

import ctypes
import os
import re

import pytest

import mla_decode_attention_gqa_gb300 as skv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "splitkv_attn.h")
SELFTEST_HEADER = os.path.join(ROOT, "include", "splitkv_attn_selftest.h")


def _declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?[\s\*]+([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_binding_symbols():
    assert _declared_functions() == sorted(skv.EXPORTED_SYMBOLS)


def test_selftest_header_declares_the_selftest_symbols():
    assert _declared_functions(SELFTEST_HEADER) == sorted(skv.SELFTEST_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = skv.load_library()
    for name in _declared_functions() + _declared_functions(SELFTEST_HEADER):
        assert hasattr(lib, name), name
    assert skv.version() == (1, 0)


def _desc(**kw):
    d = skv.SkvDesc()
    d.B, d.Tq, d.Hq, d.Hkv, d.dk, d.dv = 2, 1, 16, 4, 128, 128
    d.S_max = 1024
    d.softmax_scale = 0.088
    d.kv_dtype = skv.SKV_KV_BF16 if hasattr(skv, "SKV_KV_BF16") else 0
    d.scale_block = 64
    q = [16 * 128, 16 * 128, 128]
    k = [4 * 1024 * 128, 1024 * 128, 128]
    for i in range(3):
        d.q_strides[i], d.k_strides[i], d.v_strides[i] = q[i], k[i], k[i]
    for key, val in kw.items():
        if key in ("q_strides", "k_strides", "v_strides"):
            for i in range(3):
                getattr(d, key)[i] = val[i]
        else:
            setattr(d, key, val)
    return d


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def _call_partial(d, bounds=FAKE, n_split=1, q=FAKE, k=FAKE, v=FAKE, seq=FAKE, ks=None, vs=None):
    lib = skv.load_library()
    return lib.attn_partial(ctypes.byref(d), q, k, v, ks, vs, seq, bounds, n_split, 0, FAKE, FAKE, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=15), skv.SKV_EINVAL),
    (dict(B=0), skv.SKV_EINVAL),
    (dict(S_max=0), skv.SKV_EINVAL),
    (dict(softmax_scale=float("inf")), skv.SKV_EINVAL),
    (dict(kv_dtype=7), skv.SKV_EINVAL),
    (dict(q_strides=(16 * 128, 16 * 128, 100)), skv.SKV_EINVAL),
    (dict(k_strides=(4 * 1024 * 128, 1024 * 128, 100)), skv.SKV_EINVAL),
    (dict(dk=96, dv=96), skv.SKV_EUNSUPPORTED),
    (dict(dk=128, dv=64), skv.SKV_EUNSUPPORTED),
    (dict(kv_dtype=1, scale_block=32), skv.SKV_EINVAL),
])
def test_bad_descriptors_are_rejected(kw, status):
    assert _call_partial(_desc(**kw)) == status
    assert skv.last_error() != ""


def test_bad_pointers_and_bounds_are_rejected():
    d = _desc()
    assert _call_partial(d, q=None) == skv.SKV_EINVAL
    assert _call_partial(d, seq=None) == skv.SKV_EINVAL
    assert _call_partial(d, k=ctypes.c_void_p(0x10008)) == skv.SKV_EINVAL  # not 16-byte aligned
    assert _call_partial(d, bounds=None) == skv.SKV_EINVAL  # no bounds table
    assert "split_bounds" in skv.last_error()
    assert _call_partial(d, bounds=ctypes.c_void_p(0x10002)) == skv.SKV_EINVAL  # bounds not 4-byte aligned
    assert _call_partial(d, n_split=0) == skv.SKV_EINVAL
    d8 = _desc(kv_dtype=1)
    assert _call_partial(d8) == skv.SKV_EINVAL  # fp8 without scales
    assert "scale" in skv.last_error()


def test_serving_batches_pass_host_validation():
    """The bounds table is device memory the host never reads, so the batch size is not
    capped by it: B = 4096 sequences over 8 splits (36,864 bounds) passes every host check
    and reaches the workspace check; pass-Q and ring steps take large batches too."""
    lib = skv.load_library()
    d = _desc(B=4096)
    assert skv.gqa_decode_attn_workspace_size(d, 8) > 0
    st = lib.gqa_decode_attn(ctypes.byref(d), FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 8, 0, FAKE, FAKE, None, 0,
                             None)
    assert st == skv.SKV_EWORKSPACE, skv.last_error()
    n = ctypes.c_size_t(0)
    assert lib.attn_ring_step_workspace_size(ctypes.byref(_desc(B=2048)), ctypes.byref(n)) == skv.SKV_OK
    assert lib.gqa_decode_attn_passq_workspace_size(ctypes.byref(_desc(B=1024)), 4, ctypes.byref(n)) == skv.SKV_OK


def test_merge_argument_checks():
    lib = skv.load_library()
    assert lib.attn_merge_lse(0, 1, 1, 1, 4, FAKE, FAKE, FAKE, FAKE, None) == skv.SKV_EINVAL
    assert lib.attn_merge_lse(2, 1, 1, 1, 6, FAKE, FAKE, FAKE, FAKE, None) == skv.SKV_EINVAL
    assert lib.attn_merge_lse(2, 1, 1, 1, 8, None, FAKE, FAKE, FAKE, None) == skv.SKV_EINVAL


def test_workspace_sizes_are_host_queries():
    d = _desc()
    assert skv.gqa_decode_attn_workspace_size(d, 1) > 0
    assert skv.attn_partial_workspace_size(d, 1) >= 0
    # the tensor-core shapes (bf16 d = 128, >= 128 rows per KV head) merge in the kernel
    assert skv.gqa_decode_attn_workspace_size(_desc(Tq=32, q_strides=(32 * 16 * 128, 16 * 128, 128)), 4) == 0


def test_missing_workspace_is_reported():
    lib = skv.load_library()
    d = _desc()
    st = lib.gqa_decode_attn(ctypes.byref(d), FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 1, 0, FAKE, FAKE, None, 0,
                             None)
    assert st == skv.SKV_EWORKSPACE


def _paged(block_len=64, max_blocks=16, num_blocks=40, table=FAKE):
    pg = skv.SkvPaged()
    pg.block_len, pg.max_blocks, pg.num_blocks = block_len, max_blocks, num_blocks
    pg.block_table = table.value if table is not None else None
    return pg


def _call_paged(d, pg):
    lib = skv.load_library()
    return lib.attn_partial_paged(ctypes.byref(d), ctypes.byref(pg) if pg is not None else None, FAKE, FAKE, FAKE,
                                  None, None, FAKE, FAKE, 1, 0, FAKE, FAKE, None, 0, None)


def test_paged_arguments_are_checked_before_any_device_access():
    d = _desc()  # S_max = 1024
    assert _call_paged(d, None) == skv.SKV_EINVAL
    assert _call_paged(d, _paged(block_len=96)) == skv.SKV_EINVAL  # not a multiple of 64
    assert "block_len" in skv.last_error()
    assert _call_paged(d, _paged(block_len=0)) == skv.SKV_EINVAL
    assert _call_paged(d, _paged(table=None)) == skv.SKV_EINVAL
    assert _call_paged(d, _paged(table=ctypes.c_void_p(0x10002))) == skv.SKV_EINVAL  # misaligned
    assert _call_paged(d, _paged(max_blocks=8)) == skv.SKV_EINVAL  # 8 * 64 < S_max
    assert "S_max" in skv.last_error()
    assert _call_paged(d, _paged(num_blocks=0)) == skv.SKV_EINVAL
    d8 = _desc(kv_dtype=1, scale_block=128)
    assert _call_paged(d8, _paged(block_len=64)) == skv.SKV_EINVAL  # pages smaller than a scale block


def test_position_arguments_are_checked_before_any_device_access():
    lib = skv.load_library()

    def call(d, qp, kp):
        return lib.attn_partial_pos(ctypes.byref(d), FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 1, qp, kp, FAKE, FAKE,
                                    None, 0, None)

    d = _desc()
    assert call(d, None, FAKE) == skv.SKV_EINVAL
    assert call(d, FAKE, None) == skv.SKV_EINVAL
    assert call(d, FAKE, ctypes.c_void_p(0x10004)) == skv.SKV_EINVAL  # k_pos not 16-byte aligned
    assert call(_desc(S_max=1022), FAKE, FAKE) == skv.SKV_EINVAL  # S_max not a multiple of 4
    mla = _desc(Hq=128, Hkv=1, dk=576, dv=512, q_strides=(128 * 576, 128 * 576, 576),
                k_strides=(1024 * 576, 1024 * 576, 576), v_strides=(1024 * 576, 1024 * 576, 576))
    assert call(mla, FAKE, FAKE) == skv.SKV_EUNSUPPORTED


def test_ring_step_arguments_are_checked():
    lib = skv.load_library()
    d = _desc()
    n = ctypes.c_size_t(0)
    assert lib.attn_ring_step_workspace_size(ctypes.byref(d), ctypes.byref(n)) == skv.SKV_OK and n.value > 0
    st = lib.attn_ring_step(ctypes.byref(d), FAKE, FAKE, FAKE, None, None, FAKE, 0, 0, None, FAKE, FAKE, n.value, None)
    assert st == skv.SKV_EINVAL  # no o_acc
    st = lib.attn_ring_step(ctypes.byref(d), FAKE, FAKE, FAKE, None, None, FAKE, 0, 0, FAKE, FAKE, None, 0, None)
    assert st == skv.SKV_EWORKSPACE  # a later step needs its workspace
    assert lib.attn_ring_step_workspace_size(ctypes.byref(_desc(B=0)), ctypes.byref(n)) == skv.SKV_EINVAL


def test_passq_arguments_are_checked():
    lib = skv.load_library()
    n = ctypes.c_size_t(0)

    def ws(d, n_ranks):
        return lib.gqa_decode_attn_passq_workspace_size(ctypes.byref(d), n_ranks, ctypes.byref(n))

    assert ws(_desc(B=4), 2) == skv.SKV_OK and n.value > 0
    assert ws(_desc(B=3), 2) == skv.SKV_EINVAL  # B not a multiple of the group
    assert ws(_desc(B=4), 0) == skv.SKV_EINVAL
    assert ws(_desc(B=4, Tq=2), 2) == skv.SKV_EUNSUPPORTED  # decode only
    mla = _desc(B=4, Hq=128, Hkv=1, dk=576, dv=512, q_strides=(128 * 576, 128 * 576, 576),
                k_strides=(1024 * 576, 1024 * 576, 576), v_strides=(1024 * 576, 1024 * 576, 576))
    assert ws(mla, 2) == skv.SKV_EUNSUPPORTED
    d = _desc(B=4)
    assert ws(d, 2) == skv.SKV_OK
    need = n.value
    st = lib.gqa_decode_attn_passq(ctypes.byref(d), 2, FAKE, FAKE, FAKE, None, None, FAKE, None, FAKE, FAKE, need,
                                   None)
    assert st == skv.SKV_EINVAL  # no out
    st = lib.gqa_decode_attn_passq(ctypes.byref(d), 2, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE,
                                   need - 1, None)
    assert st == skv.SKV_EWORKSPACE
    st = lib.gqa_decode_attn_passq(ctypes.byref(d), 2, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, FAKE, need,
                                   None)
    assert st == skv.SKV_EINVAL  # no shard_lens


# ---------------------------------------------------------------- binding argument checks


def test_binding_checks_caller_buffers():
    """Caller outputs must match exactly (shape, dtype, contiguous, device) before any
    pointer reaches the library; a workspace tensor is sized in bytes."""
    import torch

    dev = torch.device("cpu")
    ok = torch.empty((2, 3), dtype=torch.float32)
    assert skv._out(ok, (2, 3), torch.float32, dev, "o") is ok
    assert tuple(skv._out(None, (4,), torch.bfloat16, dev, "o").shape) == (4,)
    for bad in (torch.empty((3, 2), dtype=torch.float32), torch.empty((2, 3), dtype=torch.float64),
                torch.empty((3, 2), dtype=torch.float32).t()):
        with pytest.raises(ValueError):
            skv._out(bad, (2, 3), torch.float32, dev, "o")
    ws, nbytes = skv._ws_arg(torch.empty(10, dtype=torch.float32), 999, dev)
    assert nbytes == 40
    with pytest.raises(ValueError):
        skv._ws_arg(torch.empty((4, 4), dtype=torch.uint8).t(), 1, dev)


def test_binding_checks_lengths_and_scales():
    import torch

    skv._check_lens(torch.zeros(3, dtype=torch.int32), 3, "seq_lens")
    for bad in (torch.zeros(3, dtype=torch.int64), torch.zeros(4, dtype=torch.int32),
                torch.zeros(6, dtype=torch.int32)[::2]):
        with pytest.raises(ValueError):
            skv._check_lens(bad, 3, "seq_lens")
    skv._check_scales((torch.ones((2, 1, 5)), None), (2, 1, 5), "[B, Hkv, n]")
    with pytest.raises(ValueError):
        skv._check_scales((torch.ones((2, 1, 4)),), (2, 1, 5), "[B, Hkv, n]")


def test_binding_rejects_cpu_tensors_before_the_library():
    import torch

    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    k = torch.zeros((1, 2, 64, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        skv.gqa_decode_attn(q, k, k, torch.zeros(1, dtype=torch.int32), [[0, 64]])
    with pytest.raises(ValueError, match="CUDA tensors only"):
        skv.gqa_decode_attn(q=q, k_cache=k, v_cache=k, seq_lens=torch.zeros(1, dtype=torch.int32),
                            split_bounds=[[0, 64]])
