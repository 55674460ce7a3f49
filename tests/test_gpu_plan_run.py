"""One plan, many runs: pkv_attention_plan + pkv_paged_attention_run against
the one-call entry point (bit for bit) and against the oracle, over several
layers' pools; a run over a workspace planned for another shape; and the
stream-order regression: lengths rewritten by a GPU kernel right before every
call, many calls back to back on one stream, small block sizes (GPU required).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits, to_device_bf16

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


def _oracle_pools(w):
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    assert oracle.copy_blocks(k, v, w.cow) == 0
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0
    assert oracle.kv_append(k, v, w.k_new, w.v_new, slots) == 0
    return k, v


def _close(bits, ref, what):
    g = wl.bf16_bits_to_f32(bits).astype(np.float64)
    assert np.isfinite(g).all(), what
    err = np.abs(g - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref)), f"{what}: max err {err.max():.3e}"


def _scaled_bits(bits, e):
    """bf16 bit patterns times 2^e (exact for the N(0,1) data here; NaN stays NaN)."""
    f = wl.bf16_bits_to_f32(bits) * np.float32(2.0 ** e)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("name", ["tiny", "decode", "mix", "spec", "long"])
def test_plan_then_run_equals_one_call(name):
    w = wl.SMALL[name]()
    ds = DeviceStep(w)
    ds.cache_ops()
    ds.attention()                       # plan + run in one call
    ref = bf16_to_bits(ds.out)
    ds.out.fill_(float("nan"))
    ds.plan()
    ds.run()
    ds.run()                             # a second run over the same plan
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
    assert np.array_equal(bf16_to_bits(ds.out), ref)
    k, v = _oracle_pools(w)
    want, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0
    _close(ref, want, name)


@pytest.mark.parametrize("name,P", [("mix", 0), ("mix", 64), ("spec", 48), ("long", 0)])
def test_one_plan_serves_every_layer(name, P):
    """Four layers: each has its own pools (the step's pools scaled by 2^-l),
    queries and output; one plan, then per layer one run."""
    w = wl.SMALL[name]()
    ds = DeviceStep(w, partition_tokens=P)
    ds.cache_ops()
    k0, v0 = _oracle_pools(w)
    layers = []
    for l in range(4):
        kb, vb = _scaled_bits(k0, -l), _scaled_bits(v0, -l)
        qb = _scaled_bits(w.q, l % 2)
        layers.append(dict(k=kb, v=vb, q=qb, dk=to_device_bf16(kb, "cuda"), dv=to_device_bf16(vb, "cuda"),
                           dq=to_device_bf16(qb, "cuda"), out=torch.full_like(ds.out, float("nan"))))
    ds.plan()
    for L in layers:
        ds.run(out=L["out"], q=L["dq"], k_cache=L["dk"], v_cache=L["dv"])
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
    for l, L in enumerate(layers):
        want, st = oracle.attention(L["q"], L["k"], L["v"], w.block_tables, w.seq_lens, w.q_lens, w.scale)
        assert st == 0
        got = bf16_to_bits(L["out"])
        _close(got, want, f"{name} layer {l}")
        # and bit for bit the one-call result over that layer's buffers
        one = torch.empty_like(ds.out)
        pkv.paged_attention_decode(one, L["dq"], L["dk"], L["dv"], ds.block_tables, ds.seq_lens, ds.q_lens,
                                   ds.max_seq_len, w.scale, ds.workspace, partition_tokens=ds.partition_tokens,
                                   status=ds.status, max_q_len=ds.max_q_len)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_bits(one), got)


def test_run_over_a_plan_for_another_shape_writes_nan_and_reports():
    w = wl.SMALL["mix"]()
    ds = DeviceStep(w, max_seq_len=4096)
    ds.cache_ops()
    ds.plan()
    torch.cuda.synchronize()
    # same buffers, but the run claims a different bound on the lengths: the
    # workspace's plan key does not match, nothing is computed
    ds.out.zero_()
    ds.max_seq_len = 2048
    ds.run()
    torch.cuda.synchronize()
    assert int(ds.status.item()) & pkv.PKV_STATUS_BAD_PLAN
    assert np.isnan(wl.bf16_bits_to_f32(bf16_to_bits(ds.out))).all()
    # a matching plan clears it
    ds.status.zero_()
    ds.plan()
    ds.run()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    assert np.isfinite(wl.bf16_bits_to_f32(bf16_to_bits(ds.out))).all()


def test_fp8_plan_then_runs_equal_one_call():
    w = wl.SMALL["mix"]()
    ds = DeviceStep(w, fp8=wl.fp8_pools(w, 3))
    ds.cache_ops()
    ds.attention()
    ref = bf16_to_bits(ds.out)
    ds.out.fill_(float("nan"))
    ds.plan()
    ds.run()
    ds.run()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    assert np.array_equal(bf16_to_bits(ds.out), ref)


def _lengths_rewritten_each_call(w, reps, partition_tokens, plan_run):
    """`reps` calls back to back on one stream; before each, GPU kernels
    rewrite seq_lens, q_lens and q (copies of shifted values, then the shift
    undone by a kernel), so the planning kernel's inputs are the output of the
    kernel launched right before it."""
    ds = DeviceStep(w, partition_tokens=partition_tokens)
    ds.cache_ops()
    seq_src = (ds.seq_lens - 7).clone()
    ql_src = (ds.q_lens + 3).clone()
    q_src = (ds.q.float() * 2.0).to(torch.bfloat16)
    outs = []
    for _ in range(reps):
        ds.seq_lens.copy_(seq_src)
        ds.q_lens.copy_(ql_src)
        ds.q.copy_(q_src)
        ds.seq_lens.add_(7)              # a kernel right before the call writes the lengths
        ds.q_lens.sub_(3)
        ds.q.mul_(0.5)                   # exact in bf16
        if plan_run:
            ds.plan()
            ds.run()
        else:
            ds.attention()
        outs.append(ds.out.clone())
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
    return [bf16_to_bits(o) for o in outs]


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("kind", ["decode", "spec"])
@pytest.mark.parametrize("plan_run", [False, True])
def test_back_to_back_calls_with_lengths_written_on_the_gpu(bs, kind, plan_run):
    if kind == "decode":
        w = wl.decode(B=9, lo=1, hi=300, seed=40 + bs, n_q=8, n_kv=2, d=128, bs=bs)
    else:
        w = wl.spec(B=5, lo=8, hi=260, k=4, vocab=64, seed=50 + bs, n_q=8, n_kv=2, d=128, bs=bs)
    outs = _lengths_rewritten_each_call(w, 40, 48, plan_run)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    k, v = _oracle_pools(w)
    want, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0
    _close(outs[0], want, f"{kind} bs {bs}")


@pytest.mark.parametrize("name", ["decode", "mix", "spec", "tiny"])
def test_step_with_the_plan_on_a_side_stream(name):
    # the bench's step: in a step that copies blocks on write (mix, tiny) the
    # plan on its own stream beside the cache ops and the run after both, else
    # every kernel in order on the main stream; every step bit-identical to the
    # one-stream step, and the first within tolerance of the oracle
    w = wl.SMALL[name]()
    ds = DeviceStep(w)
    assert ds.plan_beside_cache_ops() == (name in ("mix", "tiny"))
    ds.step()
    torch.cuda.synchronize()
    ref = bf16_to_bits(ds.out)
    k, v = _oracle_pools(w)
    want, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0
    _close(ref, want, name)
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    for _ in range(5):
        ds.reset_cache()
        ds.out.fill_(float("nan"))
        ds.step(main, side)
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
    assert np.array_equal(bf16_to_bits(ds.out), ref)
