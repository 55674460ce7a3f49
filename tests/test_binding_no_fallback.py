"""The product path has no CPU fallback: the binding refuses host tensors,
non-contiguous tensors and wrong dtypes with an error before any work is
enqueued (CPU test, no GPU needed)."""
import pytest
import torch

import paged_kv_cache_23_gb300 as pkv


def _attention_args(device="cpu", dtype=torch.bfloat16):
    nb, n_kv, bs, d, n_q = 4, 2, 16, 64, 4
    kc = torch.zeros(nb, n_kv, bs, d, dtype=dtype, device=device)
    return dict(out=torch.zeros(1, n_q, d, dtype=dtype, device=device), q=torch.zeros(1, n_q, d, dtype=dtype, device=device),
                k_cache=kc, v_cache=kc.clone(), block_tables=torch.zeros(1, 4, dtype=torch.int32, device=device),
                seq_lens=torch.ones(1, dtype=torch.int32, device=device), q_lens=torch.ones(1, dtype=torch.int32, device=device),
                max_seq_len=64, scale=0.125, workspace=torch.zeros(256, dtype=torch.uint8, device=device))


def test_attention_refuses_host_tensors():
    with pytest.raises(pkv.PkvError, match="CUDA tensor"):
        pkv.paged_attention_decode(**_attention_args())


def test_attention_refuses_wrong_dtype_and_layout():
    a = _attention_args()
    a["q"] = a["q"].float()
    with pytest.raises(pkv.PkvError):
        pkv.paged_attention_decode(**a)
    t = torch.zeros(4, 8)[:, ::2]
    assert not t.is_contiguous()
    with pytest.raises(pkv.PkvError):
        pkv._dev(t, "t")


def test_other_entry_points_refuse_host_tensors():
    x = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(pkv.PkvError):
        pkv.wait_selftest(1000, x)
    with pytest.raises(pkv.PkvError):
        pkv.spec_accept_greedy(torch.zeros(1, 2, 8), torch.zeros(1, 1, dtype=torch.int32), x, x, x)
    with pytest.raises(pkv.PkvError):
        pkv.kv_append(torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16), torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16),
                      torch.zeros(1, 1, 64, dtype=torch.bfloat16), torch.zeros(1, 1, 64, dtype=torch.bfloat16),
                      torch.zeros(1, dtype=torch.int64))
