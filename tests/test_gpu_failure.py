"""Failure detection on the GPU without a fault: a bounded device wait on a
flag that nothing sets (the wait every attention kernel uses) gives up,
reports PKV_STATUS_TIMEOUT through the status word the host reads, and the
context stays usable for the calls that follow."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits

pytestmark = pytest.mark.gpu


def _tiny_step_matches_oracle():
    w = wl.tiny()
    ds = DeviceStep(w)
    ds.step()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    k, v = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.copy_blocks(k, v, w.cow) == 0
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert oracle.kv_append(k, v, w.k_new, w.v_new, slots) == 0
    ref, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0
    got = wl.bf16_bits_to_f32(bf16_to_bits(ds.out)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))


@pytest.mark.parametrize("limit_ms", [20, 100])
def test_bounded_wait_gives_up_and_reports(limit_ms):
    pkv.build()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pkv.wait_selftest(limit_ms * 1_000_000, status)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == pkv.PKV_STATUS_TIMEOUT     # that bit and nothing else
    assert limit_ms / 1000 * 0.9 <= dt < limit_ms / 1000 + 5.0
    # the context answers: a whole step right after is clean and matches the oracle
    _tiny_step_matches_oracle()


def test_status_bits_accumulate_until_cleared():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.wait_selftest(1_000_000, status)
    pkv.wait_selftest(1_000_000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == pkv.PKV_STATUS_TIMEOUT
    status.zero_()
    _tiny_step_matches_oracle()
    assert int(status.item()) == 0
