"""Host-side checks of the C ABI (no GPU needed): exports, schedule, RoPE table, argument errors.

Every call here either runs pure host code or must be rejected before anything is
enqueued on a device, so none of them launches a kernel.
"""
import ctypes as C
import math
import os
import re

import numpy as np
import pytest

import dsa_indexer_cross_gb300 as D
from dsa_indexer_cross_gb300 import _lib
from oracle import dsa_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_indexer_cross_gb300.build import build
    build()


def declared_functions():
    with open(os.path.join(ROOT, "include", "dsa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+|indexshare_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 15
    lib = C.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/dsa.h but not exported"
    assert set(names) == set(_lib.EXPORTED)


def test_status_strings():
    L = D.lib()
    for code, name in _lib.STATUS_NAMES.items():
        assert L.dsa_status_string(code).decode() == name


def test_donor_table_matches_oracle_and_rejects_leading_shared():
    types = ["full" if l % 4 == 0 else "shared" for l in range(78)]
    assert D.dsa_donor_table(types) == O.donor_table(types)
    rel = ["full", "full", "full", "shared", "shared", "shared", "full", "shared", "shared", "shared"]
    assert D.dsa_donor_table(rel) == O.donor_table(rel)
    with pytest.raises(D.DsaError) as e:
        D.dsa_donor_table(["shared", "full"])
    assert e.value.name == "DSA_ERR_NO_DONOR"
    with pytest.raises(D.DsaError) as e:
        D.dsa_donor_table([1, 7])
    assert e.value.name == "DSA_ERR_ARG"


def test_rope_table_matches_float64_cos_sin():
    theta, r, n = 8e6, 64, 1 << 20
    tab = D.dsa_rope_table(theta, r, n).numpy()
    f = O.rope_inv_freq(r, theta)
    for p in (0, 1, 7, 4095, 1044480, n - 1):
        ang = p * f
        np.testing.assert_array_equal(tab[p, :, 0], np.cos(ang).astype(np.float32))
        np.testing.assert_array_equal(tab[p, :, 1], np.sin(ang).astype(np.float32))


def test_index_cache_maps_layers_to_donor_buffers():
    L = D.lib()
    types = (C.c_uint8 * 8)(1, 1, 1, 0, 0, 0, 1, 0)
    bufs = (C.c_void_p * 8)(0x1000, 0x2000, 0x3000, None, None, None, 0x7000, None)
    h = C.c_void_p()
    assert L.dsa_index_cache_create(8, types, 16, 4, bufs, C.byref(h)) == 0
    want = [0x1000, 0x2000, 0x3000, 0x3000, 0x3000, 0x3000, 0x7000, 0x7000]
    assert [L.dsa_index_cache_indices(h, l) for l in range(8)] == want
    d = C.c_int32()
    assert L.dsa_index_cache_donor(h, 5, C.byref(d)) == 0 and d.value == 2
    assert L.dsa_index_cache_donor(h, 8, C.byref(d)) == 1
    assert L.dsa_index_cache_indices(h, -1) is None
    L.dsa_index_cache_destroy(h)
    # a full layer without a buffer, and a schedule with no donor, are rejected
    bufs[6] = None
    assert L.dsa_index_cache_create(8, types, 16, 4, bufs, C.byref(h)) == 1
    types2 = (C.c_uint8 * 2)(0, 1)
    assert L.dsa_index_cache_create(2, types2, 16, 4, bufs, C.byref(h)) == 3


def _idesc(**kw):
    base = dict(n_q=8, n_kv=64, n_heads=32, head_dim=128, rope_dim=64, topk=16, max_len=64,
                flags=D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    base.update(kw)
    return _lib.IndexerDesc(*base.values())


@pytest.mark.parametrize("kw,name", [
    (dict(head_dim=96), "DSA_ERR_UNSUPPORTED"),
    (dict(n_heads=48), "DSA_ERR_UNSUPPORTED"),
    (dict(rope_dim=3), "DSA_ERR_ARG"),
    (dict(rope_dim=130), "DSA_ERR_ARG"),
    (dict(topk=0), "DSA_ERR_UNSUPPORTED"),
    (dict(topk=4096), "DSA_ERR_UNSUPPORTED"),
    (dict(max_len=65), "DSA_ERR_ARG"),
    (dict(n_q=-1), "DSA_ERR_ARG"),
    (dict(flags=1 << 9), "DSA_ERR_ARG"),
])
def test_indexer_descriptor_errors(kw, name):
    with pytest.raises(D.DsaError) as e:
        D.dsa_indexer_workspace_size(_idesc(**kw))
    assert e.value.name == name


def test_indexer_null_pointers_rejected_before_launch():
    L = D.lib()
    desc = _idesc()
    st = L.dsa_indexer_topk(C.byref(desc), None, None, None, None, None, None, None, None, 0, None, None, None, 0, None)
    assert st == 1 and "non-NULL" in L.dsa_last_error().decode()
    # misaligned bf16 pointer
    st = L.dsa_indexer_topk(C.byref(desc), 0x1001, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 16,
                            0x9000, None, 0x10000, 1 << 30, None)
    assert st == 1 and "aligned" in L.dsa_last_error().decode()


def test_workspace_size_grows_with_rows_and_is_256_aligned():
    a = D.dsa_indexer_workspace_size(_idesc(n_q=64))
    b = D.dsa_indexer_workspace_size(_idesc(n_q=128))
    assert b > a and a % 256 == 0 and b % 256 == 0
    no_rope = D.dsa_indexer_workspace_size(_idesc(n_q=64, flags=0))
    assert no_rope < a


@pytest.mark.parametrize("kw,name", [
    (dict(d_qk=192), "DSA_ERR_UNSUPPORTED"),
    (dict(n_heads=0), "DSA_ERR_UNSUPPORTED"),
    (dict(n_heads=256), "DSA_ERR_UNSUPPORTED"),
    (dict(softmax_scale=0.0), "DSA_ERR_ARG"),
    (dict(softmax_scale=float("nan")), "DSA_ERR_ARG"),
    (dict(topk=0), "DSA_ERR_ARG"),
])
def test_attention_descriptor_errors(kw, name):
    base = dict(n_q=4, n_kv=16, n_heads=16, d_qk=576, d_v=512, topk=8, softmax_scale=1 / 24.0, flags=0)
    base.update(kw)
    with pytest.raises(D.DsaError) as e:
        D.dsa_sparse_attn_workspace_size(_lib.AttnDesc(*base.values()))
    assert e.value.name == name


def test_layer_loop_rejects_mismatched_schedule_before_launch():
    L = D.lib()
    types = (C.c_uint8 * 4)(1, 0, 0, 0)
    bufs = (C.c_void_p * 4)(0x1000, None, None, None)
    h = C.c_void_p()
    assert L.dsa_index_cache_create(4, types, 8, 16, bufs, C.byref(h)) == 0
    idesc = _idesc()
    adesc = _lib.AttnDesc(8, 64, 16, 576, 512, 16, 1 / 24.0, 0)
    io = (_lib.LayerIO * 4)()
    other = (C.c_uint8 * 4)(1, 0, 1, 0)
    st = L.indexshare_layers_forward(C.byref(idesc), C.byref(adesc), 4, other, io, None, None, None, None, None, 0, h,
                                     0x100000, 1 << 30, None)
    assert st == 2 and "indexer_types" in L.dsa_last_error().decode()
    adesc_bad = _lib.AttnDesc(8, 64, 16, 576, 512, 32, 1 / 24.0, 0)
    st = L.indexshare_layers_forward(C.byref(idesc), C.byref(adesc_bad), 4, types, io, None, None, None, None, None, 0,
                                     h, 0x100000, 1 << 30, None)
    assert st == 2
    L.dsa_index_cache_destroy(h)


def test_profiling_switch_and_argument_errors():
    # the switch needs no device; reading needs a non-NULL buffer of at least one value
    L = _lib.lib()
    assert L.dsa_profile_enable(1) == 0
    assert L.dsa_profile_indexer_last(None, 4) == 1          # DSA_ERR_ARG
    buf = (C.c_float * 4)()
    assert L.dsa_profile_indexer_last(buf, 0) == 1
    assert L.dsa_profile_enable(0) == 0


def test_mtp_step_argument_errors_before_launch():
    # step < 0, NULL mtp_idx, missing step-0 indexer inputs and disagreeing descriptors are
    # all rejected on the host (fake non-NULL pointers are never dereferenced)
    L = _lib.lib()
    idesc = D.indexer_desc(8, 64, 4, 64, 16, 32, 64, D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    adesc = D.attn_desc(8, 64, 4, 32, 1 / 24.0)
    fake = 0x100000
    io = _lib.LayerIO(fake, fake, fake, fake, fake, fake, None)
    args = (None, None, None, None, None, 0)
    assert L.dsa_mtp_indexshare_step(C.byref(idesc), C.byref(adesc), -1, C.byref(io), *args, fake, fake, 1 << 30,
                                     None) == 1
    assert "step" in L.dsa_last_error().decode()
    assert L.dsa_mtp_indexshare_step(C.byref(idesc), C.byref(adesc), 0, C.byref(io), *args, None, fake, 1 << 30,
                                     None) == 1
    io0 = _lib.LayerIO(None, fake, fake, fake, fake, fake, None)
    assert L.dsa_mtp_indexshare_step(C.byref(idesc), C.byref(adesc), 0, C.byref(io0), *args, fake, fake, 1 << 30,
                                     None) == 1
    assert "q_idx" in L.dsa_last_error().decode()
    adesc_bad = D.attn_desc(8, 64, 4, 16, 1 / 24.0)
    assert L.dsa_mtp_indexshare_step(C.byref(idesc), C.byref(adesc_bad), 1, C.byref(io), *args, fake, fake, 1 << 30,
                                     None) == 2


def test_paged_calls_reject_bad_layouts_before_launch():
    L = _lib.lib()
    fake = 0x100000
    flags = D.DSA_IDX_ROPE_Q | D.DSA_IDX_INDEPENDENT_ROWS
    idesc = D.indexer_desc(4, 8 * 128, 64, 128, 64, 32, 1024, flags)
    pages = _lib.PagedCache(fake, fake, 8, 8, 128)
    args = (fake, fake, fake, fake)
    ok_rest = (fake, 16, fake, None, fake, 1 << 30, None)
    bad = _lib.PagedCache(fake, fake, 8, 8, 64)                    # page_rows other than 128
    assert L.dsa_indexer_topk_paged(C.byref(idesc), *args, C.byref(bad), *ok_rest) == 4
    short = _lib.PagedCache(fake, fake, 8, 7, 128)                 # n_kv != n_pages * page_rows
    assert L.dsa_indexer_topk_paged(C.byref(idesc), *args, C.byref(short), *ok_rest) == 2
    roped = D.indexer_desc(4, 8 * 128, 64, 128, 64, 32, 1024, flags | D.DSA_IDX_ROPE_K)
    assert L.dsa_indexer_topk_paged(C.byref(roped), *args, C.byref(pages), *ok_rest) == 1
    h32 = D.indexer_desc(4, 8 * 128, 32, 128, 64, 32, 1024, flags)
    assert L.dsa_indexer_topk_paged(C.byref(h32), *args, C.byref(pages), *ok_rest) == 4
    long_ = D.indexer_desc(4, 8 * 128, 64, 128, 64, 32, 1025, flags)   # max_len beyond max_pages pages
    assert L.dsa_indexer_topk_paged(C.byref(long_), *args, C.byref(pages), *ok_rest) == 1
    nobt = _lib.PagedCache(None, fake, 8, 8, 128)
    assert L.dsa_indexer_topk_paged(C.byref(idesc), *args, C.byref(nobt), *ok_rest) == 1
    adesc = D.attn_desc(4, 8 * 128, 16, 32, 1 / 24.0)
    assert L.dsa_sparse_attn_paged(C.byref(adesc), fake, fake, fake, C.byref(short), fake, None, fake, 1 << 30,
                                   None) == 2
    assert L.dsa_sparse_attn_paged(C.byref(adesc), fake, fake, fake, None, fake, None, fake, 1 << 30, None) == 1


def test_attention_backward_argument_errors_before_launch():
    # NULL tensors, misaligned tensors, a misaligned or short status workspace and a bad
    # descriptor are rejected on the host (fake pointers are never dereferenced)
    L = _lib.lib()
    adesc = D.attn_desc(4, 256, 16, 32, 1 / 24.0)
    fake = 0x100000
    t = [fake] * 9                                  # q kv idx ks out lse d_out dq dkv
    ok = L.dsa_sparse_attn_backward
    assert ok(C.byref(adesc), *t[:8], None, fake, 256, None) == 1
    for i in (0, 1, 4, 6, 7, 8):                    # the bf16 / fp32 tensors read or written in 16-byte pieces
        bad = list(t)
        bad[i] = fake + 8
        assert ok(C.byref(adesc), *bad, fake, 256, None) == 1
        assert "aligned" in L.dsa_last_error().decode()
    assert ok(C.byref(adesc), *t, fake + 16, 256, None) == 1
    assert ok(C.byref(adesc), *t, fake, 128, None) == 6
    assert ok(C.byref(D.attn_desc(4, 256, 16, 32, 1 / 24.0, d_qk=192)), *t, fake, 256, None) == 4


def test_binding_refuses_host_tensors_and_wrong_dtypes_before_the_call():
    # the ctypes binding hands bare addresses to the library, so it refuses what a kernel would
    # misread: host tensors (every tensor argument is device memory), and for the backward
    # tensors of the wrong type or size (a bf16 dkv would be written past its end as fp32)
    import torch
    adesc = D.attn_desc(2, 8, 4, 4, 1 / 24.0)
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    args = dict(q=torch.zeros((2, 4, 576), dtype=bf), kv=torch.zeros((8, 576), dtype=bf),
                idx=torch.zeros((2, 4), dtype=i32), ks=torch.zeros(2, dtype=i32),
                out=torch.zeros((2, 4, 512), dtype=bf), lse=torch.zeros((2, 4), dtype=f32),
                d_out=torch.zeros((2, 4, 512), dtype=bf), dq=torch.zeros((2, 4, 576), dtype=f32),
                dkv=torch.zeros((8, 576), dtype=f32))
    with pytest.raises(ValueError, match="CUDA"):
        D.dsa_sparse_attn(adesc, args["q"], args["kv"], args["idx"], args["ks"], args["out"], args["lse"])
    with pytest.raises(ValueError, match="CUDA"):
        D.dsa_sparse_attn_backward(adesc, **args)
    with pytest.raises(ValueError, match="dkv: expected torch.float32"):
        D.dsa_sparse_attn_backward(adesc, **dict(args, dkv=torch.zeros((8, 576), dtype=bf)))
    with pytest.raises(ValueError, match="idx: needs at least 8"):
        D.dsa_sparse_attn_backward(adesc, **dict(args, idx=torch.zeros((2, 3), dtype=i32)))


def test_empty_batch_is_a_no_op_before_any_device_work():
    # n_q = 0 is valid: the forward calls return DSA_OK without touching a pointer or a device
    L = _lib.lib()
    idesc = D.indexer_desc(0, 128, 16, 64, 32, 8, 128, D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    assert L.dsa_indexer_topk(C.byref(idesc), *([None] * 8), 0, None, None, None, 0, None) == 0
    adesc = D.attn_desc(0, 128, 16, 8, 1 / 24.0)
    assert L.dsa_sparse_attn(C.byref(adesc), *([None] * 7), 0, None) == 0
    # a negative count is an argument error
    assert L.dsa_sparse_attn(C.byref(D.attn_desc(-1, 128, 16, 8, 1 / 24.0)), *([None] * 7), 0, None) == 1


def test_forward_wrappers_check_types_and_sizes_before_the_call():
    import torch
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    adesc = D.attn_desc(2, 8, 4, 4, 1 / 24.0)
    q, kv = torch.zeros((2, 4, 576), dtype=bf), torch.zeros((8, 576), dtype=bf)
    idx, ks = torch.zeros((2, 4), dtype=i32), torch.zeros(2, dtype=i32)
    out, lse = torch.zeros((2, 4, 512), dtype=bf), torch.zeros((2, 4), dtype=f32)
    with pytest.raises(ValueError, match="q: expected torch.bfloat16"):
        D.dsa_sparse_attn(adesc, q.float(), kv, idx, ks, out, lse)
    with pytest.raises(ValueError, match="ks: expected torch.int32"):
        D.dsa_sparse_attn(adesc, q, kv, idx, ks.long(), out, lse)
    with pytest.raises(ValueError, match="out: needs at least 4096"):
        D.dsa_sparse_attn(adesc, q, kv, idx, ks, out[:1], lse)
    idesc = D.indexer_desc(2, 8, 16, 64, 32, 4, 8, D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    args = [torch.zeros((2, 16, 64), dtype=bf), torch.zeros((8, 64), dtype=bf), torch.zeros((2, 16), dtype=f32),
            torch.zeros(2, dtype=i32), torch.zeros(8, dtype=i32), ks, ks, torch.zeros((8, 16, 2), dtype=f32),
            torch.zeros((2, 4), dtype=i32)]
    with pytest.raises(ValueError, match="w: expected torch.float32"):
        D.dsa_indexer_topk(idesc, *args[:2], args[2].to(bf), *args[3:])
    with pytest.raises(ValueError, match="idx_out: needs at least 8"):
        D.dsa_indexer_topk(idesc, *args[:8], torch.zeros((2, 3), dtype=i32))
    with pytest.raises(ValueError, match="CUDA"):                         # well-formed, but host memory
        D.dsa_indexer_topk(idesc, *args)


def test_static_paged_projection_and_mtp_wrappers_check_types_and_sizes():
    # every wrapper that hands tensors to the library checks type and size first, so a
    # mistyped or short tensor never reaches a kernel as a bare pointer
    import torch
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    idesc = D.indexer_desc(2, 8, 16, 64, 32, 4, 8, D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    ks = torch.zeros(2, dtype=i32)
    args = [torch.zeros((2, 16, 64), dtype=bf), torch.zeros((8, 64), dtype=bf), torch.zeros((2, 16), dtype=f32),
            torch.zeros(2, dtype=i32), torch.zeros(8, dtype=i32), ks, ks, torch.zeros((8, 16, 2), dtype=f32),
            torch.zeros((2, 4), dtype=i32)]
    with pytest.raises(ValueError, match="q_idx: expected torch.bfloat16"):
        D.dsa_indexer_topk_static(idesc, args[0].float(), *args[1:])
    with pytest.raises(ValueError, match="idx_out: needs at least 8"):
        D.dsa_indexer_topk_static(idesc, *args[:8], torch.zeros((2, 3), dtype=i32))
    # paged: 64 index heads, one 128-row page per row
    pdesc = D.indexer_desc(2, 256, 64, 128, 64, 4, 128, D.DSA_IDX_ROPE_Q | D.DSA_IDX_INDEPENDENT_ROWS)
    pages = D.PagedCache(8, 8, 1, 2, D.DSA_PAGE_ROWS)    # fake non-NULL addresses: never reached
    q_idx, k_cache = torch.zeros((2, 64, 128), dtype=bf), torch.zeros((256, 128), dtype=bf)
    w, q_pos, idx = torch.zeros((2, 64), dtype=f32), torch.zeros(2, dtype=i32), torch.zeros((2, 4), dtype=i32)
    rope = torch.zeros((8, 32, 2), dtype=f32)
    with pytest.raises(ValueError, match="k_cache: needs at least 32768"):
        D.dsa_indexer_topk_paged(pdesc, q_idx, k_cache[:10], w, q_pos, pages, rope, idx)
    with pytest.raises(ValueError, match="w: expected torch.float32"):
        D.dsa_indexer_topk_paged(pdesc, q_idx, k_cache, w.to(bf), q_pos, pages, rope, idx)
    adesc = D.attn_desc(2, 256, 4, 4, 1 / 24.0)
    q, kvc = torch.zeros((2, 4, 576), dtype=bf), torch.zeros((256, 576), dtype=bf)
    out = torch.zeros((2, 4, 512), dtype=bf)
    with pytest.raises(ValueError, match="idx: expected torch.int32"):
        D.dsa_sparse_attn_paged(adesc, q, kvc, idx.long(), pages, out)
    with pytest.raises(ValueError, match="kv_cache: needs at least"):
        D.dsa_sparse_attn_paged(adesc, q, kvc[:3], idx, pages, out)
    # projections
    pd = D.ProjDesc(4, 128, 64, 16, 64, 1e-6)
    t = dict(x=torch.zeros((4, 128), dtype=bf), q_latent=torch.zeros((4, 64), dtype=bf),
             wq_b=torch.zeros((1024, 64), dtype=bf), wk=torch.zeros((64, 128), dtype=bf),
             k_norm_w=torch.ones(64), k_norm_b=torch.zeros(64), weights_proj=torch.zeros((16, 128), dtype=bf),
             q_idx=torch.zeros((4, 16, 64), dtype=bf), k_idx=torch.zeros((4, 64), dtype=bf),
             w=torch.zeros((4, 16), dtype=f32))
    with pytest.raises(ValueError, match="wk: needs at least 8192"):
        D.dsa_indexer_projections(pd, **dict(t, wk=t["wk"][:3]))
    with pytest.raises(ValueError, match="k_norm_w: expected torch.float32"):
        D.dsa_indexer_projections(pd, **dict(t, k_norm_w=torch.ones(64, dtype=bf)))
    # MTP step
    layer = dict(q=q, kv=kvc, out=out, q_idx=torch.zeros((2, 16, 64), dtype=bf), k_idx=torch.zeros((256, 64), dtype=bf),
                 w=torch.zeros((2, 16), dtype=f32))
    mdesc = D.indexer_desc(2, 256, 16, 64, 32, 4, 256, D.DSA_IDX_ROPE_Q | D.DSA_IDX_ROPE_K)
    kpos = torch.zeros(256, dtype=i32)
    with pytest.raises(ValueError, match="mtp_idx: needs at least 8"):
        D.dsa_mtp_indexshare_step(mdesc, adesc, 0, layer, ks, ks, ks, kpos, rope, torch.zeros(3, dtype=i32))
    with pytest.raises(ValueError, match="q: expected torch.bfloat16"):
        D.dsa_mtp_indexshare_step(mdesc, adesc, 1, dict(layer, q=q.float()), ks, ks, ks, kpos, rope, idx)
    with pytest.raises(ValueError, match="w: expected torch.float32"):
        D.dsa_mtp_indexshare_step(mdesc, adesc, 0, dict(layer, w=layer["w"].to(bf)), ks, ks, ks, kpos, rope, idx)
