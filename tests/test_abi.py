"""The C ABI library builds for sm_103a, loads, and exports every entry point
include/msa.h declares; host-side argument validation needs no GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_paged_02_gb300 import binding
    return binding.lib()


def test_header_declares_the_path(lib):
    syms = declared_symbols()
    for name in ("msa_index_score", "msa_topk_build_table", "msa_sparse_paged_attn",
                 "msa_decode", "msa_workspace_size", "msa_status_string"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def header_structs():
    """Field names and C types of every struct typedef in include/msa.h, in order."""
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for name, body in re.findall(r"typedef struct (\w+) \{(.*?)\} \1;", src, flags=re.S):
        fields = []
        for decl in body.split(";"):
            decl = " ".join(decl.split())
            if decl:
                m = re.match(r"(.*?)(\w+)$", decl)
                fields.append((m.group(2), m.group(1).replace(" ", "")))
        out[name] = fields
    return out


def test_struct_layouts_match_header():
    # the ctypes mirrors in the binding follow the header field by field:
    # same names, same order, and a pointer / 64-bit / 32-bit / float kind
    # per field, so a field added to one side alone fails here
    from block_sparse_paged_02_gb300 import binding as B
    structs = header_structs()
    assert set(structs) == {"msa_batch", "msa_attn_args", "msa_trace", "msa_index_cache",
                            "msa_mla_args"}
    for name, fields in structs.items():
        py = getattr(B, name)._fields_
        assert [f for f, _ in fields] == [f for f, _ in py], name
        for (f, ctype), (_, pytype) in zip(fields, py):
            if "*" in ctype or ctype in ("cudaEvent_t", "cudaStream_t"):
                assert pytype is ctypes.c_void_p, (name, f)
            elif ctype == "float":
                assert pytype is ctypes.c_float, (name, f)
            elif ctype in ("int64_t", "size_t"):
                assert ctypes.sizeof(pytype) == 8, (name, f)
            else:
                assert ctype in ("int32_t", "uint32_t", "int"), (name, f, ctype)
                assert ctypes.sizeof(pytype) == 4, (name, f)


def test_status_strings(lib):
    from block_sparse_paged_02_gb300 import binding as B
    for code in range(7):
        assert B.msa_status_string(code)
    assert "NULL" in B.msa_status_string(B.MSA_ERR_NULL)


def test_workspace_size_grows_with_rows(lib):
    from block_sparse_paged_02_gb300 import binding as B
    a = B.msa_workspace_size(8, 256, 16, 16, 128, 128)
    b = B.msa_workspace_size(64, 1024, 16, 16, 128, 128)
    assert 0 < a < b
    assert B.msa_workspace_size(64, 0, 0, 16, 128, 128) > 0
    assert B.msa_workspace_size(-1, 0, 0, 16, 128, 128) == 0


def test_host_validation_without_gpu(lib):
    from block_sparse_paged_02_gb300 import binding as B
    # NULL batch / NULL args are rejected before any launch
    assert lib.msa_index_score(None, None, None, None, 1, None, None) == B.MSA_ERR_NULL
    assert lib.msa_topk_build_table(None, None, 1, 4, None, None, 32, None, None, None) == \
        B.MSA_ERR_NULL
    assert lib.msa_sparse_paged_attn(None, None, 32, None, None, 0, None, None) == B.MSA_ERR_NULL
    fake = ctypes.c_void_p(0x10000)
    idx = lambda **kw: B.msa_index_cache(**{**dict(k_cache=fake, k_scale=None, dtype=0, heads=1,
                                                    dim=128), **kw})
    b = B.msa_batch(None, None, None, None, 4, 1, 1, 10)
    assert lib.msa_index_score(ctypes.byref(b), None, ctypes.byref(idx()), None, 4, None,
                               None) == B.MSA_ERR_NULL
    b = B.msa_batch(fake, fake, fake, fake, 4, 1, 1, 10)
    st = ctypes.c_void_p(0x20000)
    score = lambda x, stride=4: lib.msa_index_score(ctypes.byref(b), fake, ctypes.byref(x), fake,
                                                    stride, st, None)
    # no index cache; unsupported index geometry or dtype; score stride below
    # the block-table width; a misaligned FP8 scale array
    assert lib.msa_index_score(ctypes.byref(b), fake, None, fake, 4, st, None) == B.MSA_ERR_NULL
    assert score(idx(heads=3)) == B.MSA_ERR_UNSUPPORTED
    assert score(idx(dim=96)) == B.MSA_ERR_UNSUPPORTED
    assert score(idx(dtype=5)) == B.MSA_ERR_DTYPE
    assert score(idx(), stride=3) == B.MSA_ERR_SHAPE
    assert score(idx(dtype=1, k_scale=ctypes.c_void_p(0x10008))) == B.MSA_ERR_SHAPE
    # table narrower than 8*topk
    assert lib.msa_topk_build_table(ctypes.byref(b), fake, 4, 4, fake, fake, 31, fake, st,
                                    None) == B.MSA_ERR_SHAPE
    # the largest sizes: topk 2048, bt_stride 16384, 4096 requests; one past
    # each is refused before any launch
    big = B.msa_batch(fake, fake, fake, fake, 16385, 1, 1, 10)
    assert lib.msa_topk_build_table(ctypes.byref(big), fake, 16385, 4, fake, fake, 32, fake, st,
                                    None) == B.MSA_ERR_UNSUPPORTED
    many = B.msa_batch(fake, fake, fake, fake, 4, 4097, 4097, 10)
    assert lib.msa_topk_build_table(ctypes.byref(many), fake, 4, 4, fake, fake, 32, fake, st,
                                    None) == B.MSA_ERR_UNSUPPORTED
    assert lib.msa_topk_build_table(ctypes.byref(b), fake, 4, 2049, fake, fake, 8 * 2049, fake,
                                    st, None) == B.MSA_ERR_UNSUPPORTED
    # attention: 2 KV heads, head_dim 64, 17 heads, bad dtype -> rejected
    def attn(**kw):
        a = dict(q=fake, num_rows=1, num_heads=16, num_kv_heads=1, head_dim=128, k_cache=fake,
                 v_cache=fake, kv_dtype=0, num_pages=1, scale_mode=0, k_scale=None,
                 v_scale=None, sinks=None, softmax_scale=0.1, out=fake, lse=fake)
        a.update(kw)
        return B.msa_attn_args(**a)
    ws = ctypes.c_void_p(0x30000)
    call = lambda a, n=1 << 30: lib.msa_sparse_paged_attn(ctypes.byref(a), fake, 32, fake, ws, n,
                                                          st, None)
    assert call(attn(num_kv_heads=2, num_heads=16)) == B.MSA_ERR_UNSUPPORTED
    assert call(attn(head_dim=64)) == B.MSA_ERR_UNSUPPORTED
    assert call(attn(num_heads=17)) == B.MSA_ERR_UNSUPPORTED
    assert call(attn(num_heads=16, num_kv_heads=3)) == B.MSA_ERR_SHAPE
    assert call(attn(kv_dtype=7)) == B.MSA_ERR_DTYPE
    assert call(attn(scale_mode=1)) == B.MSA_ERR_NULL  # scalar scales need pointers
    assert call(attn(q=ctypes.c_void_p(0x10004))) == B.MSA_ERR_SHAPE  # misaligned
    assert call(attn(), n=16) == B.MSA_ERR_WORKSPACE


def test_sinks_contract_checked_in_binding():
    import torch
    from block_sparse_paged_02_gb300 import binding as B
    B.check_sinks(None, 16)
    B.check_sinks(torch.zeros(16), 16)
    with pytest.raises(ValueError):
        B.check_sinks(torch.zeros(16, dtype=torch.float16), 16)
    with pytest.raises(ValueError):
        B.check_sinks(torch.zeros(8), 16)
    with pytest.raises(ValueError):
        B.check_sinks(torch.zeros(32)[::2], 16)


def test_mla_host_validation_without_gpu(lib):
    from block_sparse_paged_02_gb300 import binding as B
    fake = ctypes.c_void_p(0x10000)
    st = ctypes.c_void_p(0x20000)
    def args(**kw):
        a = dict(q=fake, num_rows=2, num_heads=16, dqk=576, dv=512, kv_cache=fake,
                 num_tokens=100, kv_indptr=fake, kv_indices=fake, max_tokens=64, sinks=None,
                 softmax_scale=0.1, out=fake, lse=fake)
        a.update(kw)
        return B.msa_mla_args(**a)
    call = lambda a, n=1 << 30: lib.msa_sparse_mla_decode(ctypes.byref(a), fake, n, st, None)
    assert lib.msa_sparse_mla_decode(None, fake, 0, st, None) == B.MSA_ERR_NULL
    assert call(args(dqk=128)) == B.MSA_ERR_UNSUPPORTED
    assert call(args(dv=448)) == B.MSA_ERR_UNSUPPORTED
    assert call(args(num_heads=129)) == B.MSA_ERR_UNSUPPORTED
    assert call(args(max_tokens=0)) == B.MSA_ERR_SHAPE
    assert call(args(kv_indices=None)) == B.MSA_ERR_NULL
    assert call(args(q=ctypes.c_void_p(0x10008))) == B.MSA_ERR_SHAPE
    assert call(args(num_rows=64), n=16) == B.MSA_ERR_WORKSPACE
    # up to 8 splits merge inside a cluster (no partials); more need partials
    assert B.msa_sparse_mla_workspace_size(64, 16, 2048) >= B.msa_sparse_mla_workspace_size(1, 16, 16)
    assert B.msa_sparse_mla_workspace_size(1, 16, 20000) > B.msa_sparse_mla_workspace_size(1, 16, 2048)


def test_bounded_wait_check_validation_without_gpu(lib):
    from block_sparse_paged_02_gb300 import binding as B
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: every case fails before a launch
    assert lib.msa_check_bounded_wait(None, 1000, 0, None, None) == B.MSA_ERR_NULL
    assert lib.msa_check_bounded_wait(fake, 0, 0, None, None) == B.MSA_ERR_SHAPE
    assert lib.msa_check_bounded_wait(fake, 2_000_000, 0, None, None) == B.MSA_ERR_SHAPE
    assert lib.msa_check_bounded_wait(fake, 1000, 8, None, None) == B.MSA_ERR_UNSUPPORTED
    assert lib.msa_check_bounded_wait(fake, 1000, B.MSA_CHECK_WAIT_COPY, None, None) == \
        B.MSA_ERR_NULL
    assert lib.msa_check_bounded_wait(fake, 1000, B.MSA_CHECK_WAIT_COPY, ctypes.c_void_p(0x10008),
                                      None) == B.MSA_ERR_NULL  # misaligned source

