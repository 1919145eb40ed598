"""Checkpoint files (qw_checkpoint_*): header validation, the cross-check against the tensor set a
config implies, and the parameter counts the pages print, on synthetic files written by
tests/_ckpt.py.  Host code only: no GPU needed."""
import json
import os

import numpy as np
import pytest

import qw_inputs as qi
from oracle import shapes
from _ckpt import build, model_entries

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def qw():
    from runtime_qwen3_decode_gb300 import build as b, qw as binding
    b.build()
    return binding


def cfg(qw, wl, **kw):
    wl = wl.with_(**kw) if kw else wl
    return qw.make_config(wl, 64)


def expect_error(qw, data, what, file_size=None):
    with pytest.raises(qw.QwError) as e:
        qw.Checkpoint(data, file_size)
    assert e.value.code == qw.INVALID_ARGUMENT
    assert what in str(e.value), str(e.value)


def test_tiny_checkpoint_lists_and_checks_clean(qw):
    wl = qi.WORKLOADS["tiny"]
    w = qi.make_weights(wl)
    c = qw.Checkpoint(build(model_entries(wl, w)))
    t = c.tensors()
    assert len(t) == 3 + 11 * wl.n_layers
    byname = {n: (dt, shape) for n, dt, shape, _, _ in t}
    assert byname["model.layers.1.self_attn.q_proj.weight"] == (qw.DT_BF16, (2048, 1024))
    assert byname["model.layers.0.mlp.down_proj.weight"] == (qw.DT_BF16, (1024, 3072))
    assert all(b % 8 == 0 for _, _, _, b, _ in t)
    rc, rep = c.check(cfg(qw, wl))
    assert rc == qw.OK, rep.first_problem
    exp = shapes.expected_tensors(wl.vocab, wl.hidden, wl.n_layers, wl.n_heads, wl.n_kv_heads, wl.head_dim,
                                  wl.intermediate)
    stored, logical, emb = shapes.param_counts(exp)
    assert (rep.stored_params, rep.logical_params, rep.embedding_params) == (stored, logical, emb)
    assert rep.n_tensors == len(exp) and rep.n_missing == rep.n_unexpected == rep.n_misshaped == 0
    assert rep.lm_head_copy == 1


def test_full_shape_header_counts_match_the_pages(qw):
    # header only (the 1.4 GB blob is not needed for the checks): 311 tensors and the counts of
    # "M1 - Load the weights", section "Deriving what should be there"
    g = json.load(open(os.path.join(GOLDEN, "qwen3_0p6b_tensor_set.json")))
    wl = qi.WORKLOADS["qwen3_0p6b_decode"]
    exp = shapes.expected_tensors(wl.vocab, wl.hidden, wl.n_layers, wl.n_heads, wl.n_kv_heads, wl.head_dim,
                                  wl.intermediate)
    entries = [(n, "BF16", s, 2 * int(np.prod(s))) for n, s in exp]
    head, size = build(entries, size_only=True)
    c = qw.Checkpoint(head, size)
    rc, rep = c.check(cfg(qw, wl))
    assert rc == qw.OK, rep.first_problem
    assert rep.n_tensors == g["tensor_count"] == 311
    assert rep.stored_params == g["params_stored"] == 751_632_384
    assert rep.logical_params == g["params_logical"] == 596_049_920
    assert rep.embedding_params == g["params_embedding"] == 155_582_464
    # nothing to upload from a header
    assert qw.lib().qw_checkpoint_upload(c._h, qw.ctypes.byref(cfg(qw, wl)), 256, 1 << 30, (qw.LayerWeights * 28)(),
                                         qw.ctypes.byref(qw.Weights()), None) == qw.INVALID_ARGUMENT


def test_q8_and_f32_norms_check_against_the_int8_config(qw):
    wl = qi.WORKLOADS["tiny"].with_(weight_format="int8_g32")
    w = qi.make_weights(wl)
    c = qw.Checkpoint(build(model_entries(wl, w, q8=True, f32_norms=True)))
    assert c.check(cfg(qw, wl))[0] == qw.OK
    # Q8_0 matrices do not load into a bf16-weight model
    rc, rep = c.check(cfg(qw, qi.WORKLOADS["tiny"]))
    assert rc == qw.UNSUPPORTED_SHAPE and rep.n_bad_dtype == 7 * wl.n_layers
    assert b"dtype" in rep.first_problem


def test_tied_head_absent_or_copied(qw):
    wl = qi.WORKLOADS["tiny"]
    w = qi.make_weights(wl)
    c0 = qw.Checkpoint(build(model_entries(wl, w, head=False)))
    rc, rep = c0.check(cfg(qw, wl))
    assert rc == qw.OK and rep.lm_head_copy == 0 and rep.stored_params == rep.logical_params
    L = qw.lib()
    base = L.qw_checkpoint_upload_bytes(c0._h, qw.ctypes.byref(cfg(qw, wl)))
    same = qw.Checkpoint(build(model_entries(wl, w)))  # byte-identical copy: still tied
    assert L.qw_checkpoint_upload_bytes(same._h, qw.ctypes.byref(cfg(qw, wl))) == base
    other = w["embed"].copy()
    other[0, 0] ^= 1
    diff = qw.Checkpoint(build(model_entries(wl, w, head_bytes=other.tobytes())))
    assert L.qw_checkpoint_upload_bytes(diff._h, qw.ctypes.byref(cfg(qw, wl))) > base


def test_cross_check_reports_problems(qw):
    wl = qi.WORKLOADS["tiny"]
    w = qi.make_weights(wl)
    ents = model_entries(wl, w)
    missing = [e for e in ents if e[0] != "model.layers.1.mlp.up_proj.weight"]
    rc, rep = qw.Checkpoint(build(missing)).check(cfg(qw, wl))
    assert rc == qw.UNSUPPORTED_SHAPE and rep.n_missing == 1
    assert rep.first_problem == b"missing model.layers.1.mlp.up_proj.weight"
    extra = ents + [("model.layers.0.self_attn.rotary_emb.inv_freq", "F32", (64,), bytes(256))]
    rc, rep = qw.Checkpoint(build(extra)).check(cfg(qw, wl))
    assert rc == qw.UNSUPPORTED_SHAPE and rep.n_unexpected == 1 and b"unexpected" in rep.first_problem
    # q_proj stored transposed ([H, Hq d] instead of [Hq d, H])
    bad = [(n, dt, (s[1], s[0]) if n.endswith("q_proj.weight") else s, p) for n, dt, s, p in ents]
    rc, rep = qw.Checkpoint(build(bad)).check(cfg(qw, wl))
    assert rc == qw.UNSUPPORTED_SHAPE and rep.n_misshaped == wl.n_layers
    assert rep.first_problem.startswith(b"model.layers.0.self_attn.q_proj.weight: shape [1024,2048], expected [2048,1024]")


def raw(header_text, blob_len):
    """A file of the given header text (padded to the 8-byte grid) and a zero blob."""
    return build([], header_text=header_text) + bytes(blob_len)


def _one(dt="F32", shape=(4,), nbytes=16, off=(0, 16)):
    return '{"t":{"dtype":"%s","shape":%s,"data_offsets":[%d,%d]}}' % (dt, json.dumps(list(shape)), off[0], off[1])


def test_header_invariants_fail_closed(qw):
    ok = [("a", "F32", (4,), bytes(16)), ("b", "F32", (2,), bytes(8))]
    assert len(qw.Checkpoint(build(ok)).tensors()) == 2
    # overlapping spans
    expect_error(qw, raw('{"a":{"dtype":"F32","shape":[4],"data_offsets":[0,16]},'
                         '"b":{"dtype":"F32","shape":[4],"data_offsets":[8,24]}}', 24), "overlaps")
    # a payload off the 8-byte grid
    expect_error(qw, raw(_one(dt="F16", shape=(2,), off=(2, 6)), 8), "aligned")
    # data past the end of the file
    expect_error(qw, raw(_one(off=(0, 16)), 8), "past the file")
    # span length disagreeing with shape x dtype
    expect_error(qw, raw(_one(off=(0, 12)), 16), "does not match")
    # Q8_0 with a tail group
    expect_error(qw, raw(_one(dt="Q8_0", shape=(33,), off=(0, 34)), 40), "32-element")
    # unknown dtype, unknown key, missing key, rank > 4
    expect_error(qw, raw(_one(dt="F64"), 16), "unknown dtype")
    expect_error(qw, raw('{"t":{"dtype":"F32","shape":[4],"data_offsets":[0,16],"x":1}}', 16),
                 "unexpected or repeated key")
    expect_error(qw, raw('{"t":{"dtype":"F32","shape":[4]}}', 16), "required")
    expect_error(qw, raw(_one(shape=(1, 1, 1, 1, 4)), 16), "rank")
    # duplicate names, malformed JSON, trailing bytes, negative or fractional numbers
    expect_error(qw, raw(_one()[:-1] + ',' + _one()[1:], 16), "duplicate")
    expect_error(qw, raw(_one()[:-2], 16), "expected")
    expect_error(qw, raw(_one() + "x", 16), "trailing")
    expect_error(qw, raw(_one().replace("[4]", "[-4]"), 16), "non-negative")
    expect_error(qw, raw(_one().replace("[4]", "[4.0]"), 16), "not an integer")
    # a header length larger than the file, and a file shorter than its prefix
    data = build(ok)
    expect_error(qw, b"\xff" * 8 + data[8:], "header length")
    expect_error(qw, data[:5], "short")
    # __metadata__ holds strings only
    assert qw.Checkpoint(build(ok, metadata={"format": "pt"})).tensors()[0][0] == "a"
    expect_error(qw, raw('{"__metadata__":{"format":1}}', 0), "__metadata__")
