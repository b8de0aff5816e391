"""CPU tests of the C ABI: the library loads, exports every symbol the header
declares, and its host logic (argument checks, pool sizing, workspace sizing,
page allocator) behaves as documented.  No device work is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

from speculative_verify_attention_q3kv_gb300 import _lib, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q3kv.h")


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q3kv_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "q3kv_verify_attn" in names and "q3kv_append" in names and "q3kv_alloc_pages" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(_lib.PROTOTYPES)


def test_header_constants_match_binding():
    text = open(HEADER).read()
    consts = dict((k, int(v)) for k, v in re.findall(r"#define\s+(Q3KV_[A-Z0-9_]+)\s+(-?\d+)", text))
    for k, v in consts.items():
        if hasattr(_lib, k):
            assert getattr(_lib, k) == v, k


def test_versions_and_strerror(lib):
    assert lib.q3kv_version() >= 1
    assert lib.q3kv_format_version() == 1
    assert _lib.strerror(0) == "ok"
    assert "page" in _lib.strerror(_lib.Q3KV_ERR_OUT_OF_PAGES)
    assert _lib.strerror(12345) == "unknown error"
    # every error code the header defines has its own text
    text = open(HEADER).read()
    codes = [int(v) for v in re.findall(r"#define\s+Q3KV_ERR_[A-Z_]+\s+(-?\d+)", text)]
    assert _lib.Q3KV_ERR_HOST_MEMORY in codes
    texts = [_lib.strerror(c) for c in codes]
    assert "unknown error" not in texts and len(set(texts)) == len(codes)


def test_pool_bytes():
    d = api.make_desc(16, 2, 2561)
    assert api.pool_bytes(d) == 2561 * 16 * 2 * 2 * 256 * 112
    bad = api.make_desc(16, 2, 10)
    bad.head_dim = 128
    with pytest.raises(_lib.Q3KVError) as e:
        api.pool_bytes(bad)
    assert e.value.code == _lib.Q3KV_ERR_UNSUPPORTED
    bad = api.make_desc(16, 2, 10)
    bad.num_q_heads = 12
    with pytest.raises(_lib.Q3KVError):
        api.pool_bytes(bad)
    bad = api.make_desc(0, 2, 10)
    with pytest.raises(_lib.Q3KVError) as e:
        api.pool_bytes(bad)
    assert e.value.code == _lib.Q3KV_ERR_INVALID_ARG


def test_workspace_bytes_explicit_split():
    d = api.make_desc(16, 2, 200)
    # FMA leg, 1 slot, 32774 positions in 512-position splits, 6 tokens -> 48 rows in one 64-row chunk
    n = api.workspace_bytes(d, 1, 32774, 6, _lib.Q3KV_IMPL_FMA, 512)
    splits = -(-32774 // 512)
    assert n >= 1 * 2 * splits * 64 * (256 + 2) * 4
    with pytest.raises(_lib.Q3KVError):
        api.workspace_bytes(d, 1, 1000, 6, _lib.Q3KV_IMPL_FMA, 300)     # not a page multiple
    with pytest.raises(_lib.Q3KVError) as e:
        api.workspace_bytes(d, 1, 1000, 17, _lib.Q3KV_IMPL_FMA, 256)    # more than 16 tokens
    assert e.value.code == _lib.Q3KV_ERR_INVALID_ARG


def test_allocator_lifecycle():
    a = api.Allocator(num_pages=10, num_slots=3, max_pages_per_slot=6)
    r0 = a.alloc_pages(0, 600)                     # 3 pages
    assert list(r0[:3]) == [0, 1, 2] and np.all(r0[3:] == -1)
    r1 = a.alloc_pages(1, 256)
    assert list(r1[:1]) == [3]
    r0b = a.alloc_pages(0, 700)                    # grows by 0 pages (still 3)
    assert np.array_equal(r0, r0b)
    r0c = a.alloc_pages(0, 769)                    # 4 pages
    assert list(r0c[:4]) == [0, 1, 2, 4]
    assert a.free_pages() == 5
    with pytest.raises(_lib.Q3KVError) as e:
        a.alloc_pages(2, 6 * 256 + 1)              # more than a row holds
    assert e.value.code == _lib.Q3KV_ERR_OUT_OF_PAGES
    a.alloc_pages(2, 5 * 256)                      # exactly the 5 left
    assert a.free_pages() == 0
    with pytest.raises(_lib.Q3KVError):
        a.alloc_pages(1, 2 * 256)                  # all or nothing
    assert a.free_pages() == 0
    a.free_slot(0)
    assert a.free_pages() == 4
    r1b = a.alloc_pages(1, 3 * 256)
    assert len(set(r1b[:3].tolist())) == 3 and r1b[0] == 3
    with pytest.raises(_lib.Q3KVError) as e:
        a.alloc_pages(3, 1)
    assert e.value.code == _lib.Q3KV_ERR_SLOT_RANGE
    a.close()


def test_argument_checks_launch_nothing(lib):
    d = api.make_desc(2, 2, 4)
    # zero slots / zero tokens: OK and nothing launched (null pointers accepted)
    assert lib.q3kv_append(None, ctypes.byref(d), None, None, 4, None, None, None, 0, 0, 0, None, None, 0, None) == 0
    # a layer outside the pool
    assert lib.q3kv_append(None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1, 2, None, None, 0, None) == -1
    # an unknown dtype
    assert lib.q3kv_append(None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1, 0, None, None, 7, None) == -1
    # missing pointers with real work requested
    assert lib.q3kv_append(None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1, 0, None, None, 0, None) == -1
    # verify: too many query tokens, an unknown impl, a too-small workspace
    args = [None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1000, 17, 0, None, 0, None, 1, 256, None, 0, None]
    assert lib.q3kv_verify_attn(*args) == _lib.Q3KV_ERR_UNSUPPORTED
    args[10] = 4
    args[15] = 9
    assert lib.q3kv_verify_attn(*args) == _lib.Q3KV_ERR_INVALID_ARG
    buf = (ctypes.c_uint8 * 64)()
    addr = ctypes.addressof(buf)
    fake = (addr + 15) // 16 * 16
    args[15] = 1
    args[2] = args[3] = args[5] = args[6] = args[7] = args[12] = args[14] = fake
    assert lib.q3kv_verify_attn(*args) == _lib.Q3KV_ERR_WORKSPACE_TOO_SMALL


def test_accept_argument_checks():
    from speculative_verify_attention_q3kv_gb300 import _lib
    lib = _lib.load()
    n = ctypes.c_size_t()
    assert lib.q3kv_accept_workspace_bytes(-1, 100, ctypes.byref(n)) == _lib.Q3KV_ERR_INVALID_ARG
    assert lib.q3kv_accept_workspace_bytes(4, 0, ctypes.byref(n)) == _lib.Q3KV_ERR_INVALID_ARG
    assert lib.q3kv_accept_workspace_bytes(4, 100, None) == _lib.Q3KV_ERR_INVALID_ARG
    args = [None, 16, _lib.Q3KV_BF16, 100, 16, 16, 16, 1, 4, 4, 16, 16, 16, 16, 16, 64, None]
    bad_dtype = list(args); bad_dtype[2] = 7
    assert lib.q3kv_accept_greedy(*bad_dtype) == _lib.Q3KV_ERR_INVALID_ARG
    bad_vocab = list(args); bad_vocab[3] = 0
    assert lib.q3kv_accept_greedy(*bad_vocab) == _lib.Q3KV_ERR_INVALID_ARG
    wide = list(args); wide[9] = 17
    assert lib.q3kv_accept_greedy(*wide) == _lib.Q3KV_ERR_UNSUPPORTED
    many_rows = list(args); many_rows[8] = 70000
    assert lib.q3kv_accept_greedy(*many_rows) == _lib.Q3KV_ERR_UNSUPPORTED


def test_fp8_argument_checks(lib):
    d = api.make_desc(2, 2, 4)
    n = ctypes.c_size_t()
    assert lib.q3kv_fp8_pool_bytes(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == 4 * 2 * 2 * 2 * 256 * 256            # 256-byte records
    assert lib.q3kv_fp8_append(None, ctypes.byref(d), None, None, 4, None, None, None, 0, 0, 0, None, None, 0,
                               None) == 0
    assert lib.q3kv_fp8_append(None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1, 2, None, None, 0,
                               None) == -1
    # the CUDA-core leg does not read this format
    args = [None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1000, 4, 0, None, 0, None,
            _lib.Q3KV_IMPL_FMA, 256, None, 0, None]
    assert lib.q3kv_fp8_verify_attn(*args) == _lib.Q3KV_ERR_UNSUPPORTED


def test_nucleus_argument_checks(lib):
    i = ctypes.c_int32(0)
    p = ctypes.byref(i)
    for top_p in (0.0, -0.5, 1.5, float("nan")):
        assert lib.q3kv_accept_sample_nucleus(None, p, 0, 100, p, p, p, 1, 1, 1, p, 1.0, top_p, p, 1,
                                              p, p, p, None, 0, None) == _lib.Q3KV_ERR_INVALID_ARG


def test_prefill_and_t5k_host_checks(lib):
    d = api.make_desc(2, 2, 40)
    # prefill: the token bound is 8,192 (the verify call keeps 16); explicit splits need no device
    n_small = api.prefill_workspace_bytes(d, 1, 9000, 1000, _lib.Q3KV_IMPL_FMA, 256)
    n_big = api.prefill_workspace_bytes(d, 1, 9000, 8192, _lib.Q3KV_IMPL_FMA, 256)
    assert 0 < n_small < n_big
    with pytest.raises(_lib.Q3KVError) as e:
        api.prefill_workspace_bytes(d, 1, 9000, 8193, _lib.Q3KV_IMPL_FMA, 256)
    assert e.value.code == _lib.Q3KV_ERR_INVALID_ARG
    # turbo5k pool: 164-byte K and 112-byte V records per (page, layer, head, row)
    n = ctypes.c_size_t()
    assert lib.q3kv_t5k_pool_bytes(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == 40 * 2 * 2 * 256 * (164 + 112)
    # the turbo5k cache is read by both legs: with null buffers the tensor-core leg's call gets
    # past the plan and stops at the pointer checks instead of being refused
    args = [None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1000, 4, 0, None, 0, None,
            _lib.Q3KV_IMPL_MMA, 256, None, 0, None]
    assert lib.q3kv_t5k_verify_attn(*args) == _lib.Q3KV_ERR_INVALID_ARG
    assert lib.q3kv_t5k_append(None, ctypes.byref(d), None, None, 4, None, None, None, 1, 1, 5, None, None, 0,
                               None) == _lib.Q3KV_ERR_INVALID_ARG        # a layer outside the pool


def test_build_flags_and_dependencies():
    from speculative_verify_attention_q3kv_gb300 import build as b
    # one sm_103a target; IEEE division and no fast-math (the codec's codes are bit-exact)
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("fast" in f for f in b.NVFLAGS)
    # every file in csrc (and the public header) triggers a rebuild when it changes
    deps = set(b.dependencies())
    assert {os.path.join(b.CSRC, f) for f in os.listdir(b.CSRC)} <= deps
    assert HEADER in deps


def _c_prototypes():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for ret, name, args in re.findall(r"Q3KV_API\s+([\w\s\*]+?)\s*\b(q3kv_\w+)\s*\((.*?)\)\s*;", text, flags=re.S):
        args = " ".join(args.split())
        out[name] = (" ".join(ret.split()), [] if args in ("", "void") else [a.strip() for a in args.split(",")])
    return out


def _ctype_class(decl):
    """ctypes class(es) that can carry a C parameter declaration."""
    if "*" in decl:
        return "pointer"
    t = decl.replace("const ", "").split()[0]
    return {"int": ctypes.c_int32, "int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
            "float": ctypes.c_float, "uint64_t": ctypes.c_uint64}[t]


def test_binding_prototypes_match_the_header():
    protos = _c_prototypes()
    assert set(protos) == set(_lib.PROTOTYPES)
    for name, (ret, args) in protos.items():
        res, argtypes = _lib.PROTOTYPES[name]
        assert len(argtypes) == len(args), name
        for decl, ct in zip(args, argtypes):
            want = _ctype_class(decl)
            if want == "pointer":
                assert ct in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(ct, ctypes._Pointer), (name, decl)
            else:
                assert ct is want, (name, decl, ct)
        if ret == "void":
            assert res is None, name
        elif "char" in ret:
            assert res is ctypes.c_char_p, name
        else:
            assert res is ctypes.c_int32 and ret == "int", (name, ret)
