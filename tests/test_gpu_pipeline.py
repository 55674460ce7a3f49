"""Launch-ordering and fused-entry checks (GPU required): the fused slot
mapping + append equals the two separate calls byte for byte, and
back-to-back attention calls that share one workspace on one stream (the
planning kernel of a call overlaps the previous kernel) give the same
results as separate, synchronised calls."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


@pytest.mark.parametrize("make", [lambda: wl.SMALL["mix"](), lambda: wl.SMALL["spec"](), lambda: wl.SMALL["long"](),
                                  lambda: wl.decode(2100, 3, 40, 5, n_q=4, n_kv=2, d=64, bs=8)])
def test_fused_append_equals_two_calls(make):
    w = make()
    dev = torch.device("cuda")
    a = DeviceStep(w)
    b = DeviceStep(w)
    n = a.n_slots
    pkv.kv_append_paged(a.k_cache, a.v_cache, a.k_new, a.v_new, a.block_tables, a.seq_lens, a.append_lens, a.slots,
                        status=a.status)
    pkv.slot_mapping(b.slots, b.block_tables, b.seq_lens, b.append_lens, w.block_size, w.num_blocks, status=b.status)
    pkv.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slots, status=b.status)
    torch.cuda.synchronize()
    assert torch.equal(a.slots, b.slots)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))
    assert int(a.status.item()) == int(b.status.item()) == 0
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert np.array_equal(a.slots.cpu().numpy(), slots)


def _out(ds):
    return bf16_to_bits(ds.out).copy()


@pytest.mark.parametrize("P", [0, 4096])
def test_back_to_back_calls_share_workspace(P):
    """Two different batches through one workspace, enqueued without a
    synchronisation between them (P = 4096 leaves every row in one partition,
    the case where the attention kernel is followed by a no-op combine)."""
    w1 = wl.SMALL["mix"]()
    w2 = wl.SMALL["decode"]()
    ref = []
    for w in (w1, w2):
        ds = DeviceStep(w, partition_tokens=P or None, max_seq_len=2048)
        ds.cache_ops()
        ds.attention()
        torch.cuda.synchronize()
        ref.append((ds, _out(ds)))
    d1, d2 = ref[0][0], ref[1][0]
    # reuse one workspace for both, back to back, several times
    d2.workspace = d1.workspace
    for _ in range(5):
        d1.out.zero_()
        d2.out.zero_()
        d1.attention()
        d2.attention()
        d1.attention()
    torch.cuda.synchronize()
    assert np.array_equal(_out(d1), ref[0][1])
    assert np.array_equal(_out(d2), ref[1][1])
