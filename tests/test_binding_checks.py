"""Argument checks of the Python binding (no device work).

The C ABI takes raw device pointers, so the binding refuses, before any call
into the library, tensors the kernels could not address safely: host tensors,
tensors on another device, wrong element types, and buffers shorter than the
call's counts.  Host tensors are refused with the real library loaded.  The
shape / type / size rules are exercised with the device lookup replaced (every
tensor reads as one on device 0) and the library replaced by a recorder, so no
call with these host tensors ever reaches the library.
"""
import pytest
import torch

from speculative_verify_attention_q3kv_gb300 import _lib, api

i32 = torch.int32


class _Recorder:
    """Stands in for the loaded library: every q3kv_* call is recorded and returns 0."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return 0
        return call


@pytest.fixture
def fake(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(_lib, "load", lambda: rec)
    monkeypatch.setattr(api, "_device_index", lambda t: 0)
    monkeypatch.setattr(api, "_current_device", lambda: 0)
    monkeypatch.setattr(api, "_stream", lambda s: 0)
    return rec


def _cache(num_slots=2, rows=5, dtype=torch.bfloat16):
    desc = api.make_desc(1, 2, 8)
    return dict(desc=desc, pool=torch.zeros(64, dtype=torch.uint8),
                page_table=torch.full((num_slots, 4), -1, dtype=i32),
                lens=torch.zeros(num_slots, dtype=i32), counts=torch.zeros(num_slots, dtype=i32),
                offs=torch.zeros(num_slots + 1, dtype=i32), k=torch.zeros((rows, 2, 256), dtype=dtype),
                v=torch.zeros((rows, 2, 256), dtype=dtype), q=torch.zeros((rows, 16, 256), dtype=dtype),
                out=torch.zeros((rows, 16, 256), dtype=torch.float32), ws=torch.zeros(16, dtype=torch.uint8),
                status=torch.zeros(1, dtype=i32))


def _append(c, **kw):
    a = dict(c, **kw)
    api.append(a["desc"], a["pool"], a["page_table"], a["lens"], a["counts"], a["offs"], 3, 0, a["k"], a["v"],
               a["status"])


def _verify(c, fn=None, **kw):
    a = dict(c, **kw)
    (fn or api.verify_attn)(a["desc"], a["pool"], a["page_table"], a["lens"], a["counts"], a["offs"], 100, 3, 0,
                            a["q"], a["out"], a["ws"], 0, 0, a["status"])


def test_host_tensors_are_refused_before_any_library_call():
    c = _cache()
    with pytest.raises(ValueError, match="CUDA tensor"):
        _append(c)
    with pytest.raises(ValueError, match="CUDA tensor"):
        _verify(c)
    lg = torch.zeros((5, 100))
    z = torch.zeros(2, dtype=i32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.accept_greedy(lg, z, z, torch.zeros(5, dtype=i32), 3, z, z, z, z, None)


def test_valid_calls_reach_the_library_once(fake):
    c = _cache()
    _append(c)
    _verify(c)
    api.fp8_append(c["desc"], c["pool"], c["page_table"], c["lens"], c["counts"], c["offs"], 3, 0, c["k"], c["v"])
    _verify(c, fn=api.t5k_verify_attn)
    names = [n for n, _ in fake.calls if not n.endswith("pool_bytes")]
    assert names == ["q3kv_append", "q3kv_verify_attn", "q3kv_fp8_append", "q3kv_t5k_verify_attn"]
    args = [a for n, a in fake.calls if n == "q3kv_verify_attn"][0]
    assert args[4] == 4 and args[8] == 2             # max_pages_per_slot, num_slots from the tensors


def test_cache_call_rules(fake, monkeypatch):
    c = _cache()
    with pytest.raises(TypeError, match="int32"):
        _append(c, page_table=c["page_table"].long())
    with pytest.raises(ValueError, match="page_table"):
        _append(c, page_table=torch.zeros(8, dtype=i32))
    with pytest.raises(ValueError, match="page_table"):
        _append(c, page_table=torch.zeros((1, 4), dtype=i32))           # fewer rows than slots
    with pytest.raises(ValueError, match="one-dimensional"):
        _append(c, lens=torch.zeros((2, 1), dtype=i32))
    with pytest.raises(ValueError, match="token counts"):
        _append(c, counts=torch.zeros(1, dtype=i32))
    with pytest.raises(ValueError, match="row offsets"):
        _append(c, offs=torch.zeros(1, dtype=i32))
    with pytest.raises(TypeError, match="status"):
        _append(c, status=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match="status"):
        _append(c, status=torch.zeros(0, dtype=i32))
    with pytest.raises(TypeError, match="share a dtype"):
        _append(c, v=c["v"].float())
    with pytest.raises(ValueError, match=r"\[rows, 2, 256\]"):
        _append(c, k=torch.zeros((5, 3, 256), dtype=torch.bfloat16), v=torch.zeros((5, 3, 256), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="differ in shape"):
        _append(c, v=torch.zeros((4, 2, 256), dtype=torch.bfloat16))
    monkeypatch.setattr(api, "pool_bytes", lambda d: 65)
    with pytest.raises(ValueError, match="pool holds 64 bytes"):
        _append(c)
    assert not [n for n, _ in fake.calls if not n.endswith("pool_bytes")]


def test_verify_call_rules(fake):
    c = _cache()
    with pytest.raises(TypeError, match="float32"):
        _verify(c, out=c["out"].half())
    with pytest.raises(ValueError, match=r"\[rows, 16, 256\]"):
        _verify(c, q=torch.zeros((5, 8, 256), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out has 4 rows"):
        _verify(c, out=torch.zeros((4, 16, 256)))
    with pytest.raises(ValueError, match="lengths"):
        _verify(c, lens=None)
    _verify(c, out=torch.zeros((9, 16, 256)))                             # a longer output buffer is fine
    c0 = _cache(num_slots=0, rows=0)
    _verify(c0, page_table=torch.zeros((0, 1), dtype=i32))                 # an empty call passes through
    assert [n for n, _ in fake.calls if not n.endswith("pool_bytes")] == ["q3kv_verify_attn"] * 2


def test_other_device_is_refused(fake, monkeypatch):
    c = _cache()
    other = c["q"]
    monkeypatch.setattr(api, "_device_index", lambda t: 1 if t is other else 0)
    with pytest.raises(ValueError, match="cuda:1"):
        _verify(c)


def test_accept_call_rules(fake):
    lg = torch.zeros((5, 100), dtype=torch.bfloat16)
    z = torch.zeros(2, dtype=i32)
    toks = torch.zeros(5, dtype=i32)
    u = torch.zeros(5)
    api.accept_greedy(lg, z, z, toks, 3, z, z, z, z, None)
    api.accept_sample(lg, z, z, toks, 3, z, 1.0, u, 1, z, z, z, None)
    api.accept_sample_nucleus(lg, z, z, toks, 3, z, 1.0, 0.9, u, 1, z, z, z, None)
    assert [n for n, _ in fake.calls] == ["q3kv_accept_greedy", "q3kv_accept_sample", "q3kv_accept_sample_nucleus"]
    with pytest.raises(ValueError, match=r"\[rows, vocab\]"):
        api.accept_greedy(lg.flatten(), z, z, toks, 3, z, z, z, z, None)
    with pytest.raises(TypeError, match="float32 or bfloat16"):
        api.accept_greedy(lg.half(), z, z, toks, 3, z, z, z, z, None)
    with pytest.raises(ValueError, match="tokens"):
        api.accept_greedy(lg, z, z, toks[:4], 3, z, z, z, z, None)
    with pytest.raises(ValueError, match="committed_len"):
        api.accept_greedy(lg, z, z, toks, 3, z, z, z, z[:1], None)
    with pytest.raises(TypeError, match="n_accepted"):
        api.accept_greedy(lg, z, z, toks, 3, z, z.long(), z, z, None)
    with pytest.raises(TypeError, match="uniforms"):
        api.accept_sample(lg, z, z, toks, 3, z, 1.0, u.double(), 1, z, z, z, None)
    with pytest.raises(ValueError, match="uniforms"):
        api.accept_sample_nucleus(lg, z, z, toks, 3, z, 1.0, 0.9, u[:3], 1, z, z, z, None)
    assert len(fake.calls) == 3


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no library and no build: the binding raises; there is no other path to the results
    from speculative_verify_attention_q3kv_gb300 import build as b
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(b, "LIB", str(tmp_path / "libq3kv.so"))
    with pytest.raises(OSError, match="libq3kv.so not found"):
        _lib.load(build_if_missing=False)
    monkeypatch.setattr(b, "build", lambda *a, **k: (_ for _ in ()).throw(RuntimeError("nvcc not found")))
    with pytest.raises(RuntimeError, match="nvcc"):
        api.pool_bytes(api.make_desc(1, 2, 8))
