"""Host-side input generators (CPU): the paged layout and the packed-sequence
offsets the GPU tests rely on, checked against the contiguous tensors they come from."""

import torch

from exact_attention_43_gb300 import workloads as wl


def test_paged_cache_reassembles_the_contiguous_cache():
    lens = [37, 0, 64, 5]
    q, k, v, _ = wl.decode_inputs(4, 4, 2, 64, 16, torch.tensor(lens), seed=7)
    for page in (1, 7, 16, 64, 100):
        kp, vp, table = wl.paged_cache(k, v, lens, page, seed=8)
        assert table.dtype == torch.int32 and table.shape == (4, -(-64 // page))
        used = table[table >= 0]
        assert len(set(used.tolist())) == used.numel()              # no page shared
        assert int(used.max()) < kp.shape[0]
        for b, L in enumerate(lens):
            n = -(-L // page)
            assert bool((table[b, n:] == -1).all())                   # entries past the pages
            for j in range(L):
                pg, off = divmod(j, page)
                phys = int(table[b, pg])
                assert torch.equal(kp[phys, :, off], k[b, :, j])
                assert torch.equal(vp[phys, :, off], v[b, :, j])


def test_varlen_inputs_offsets_and_padding():
    lq, lk = [3, 0, 5], [4, 2, 0]
    q, k, v, cq, ck = wl.varlen_inputs(lq, lk, 4, 2, 8, seed=9, pad_q=2)
    assert cq.tolist() == [0, 3, 3, 8] and ck.tolist() == [0, 4, 6, 6]
    assert q.shape == (8 + 2, 4, 8) and k.shape == (6, 2, 8) and v.shape == k.shape
    # seeded: the same call gives the same tensors
    q2, k2, v2, _, _ = wl.varlen_inputs(lq, lk, 4, 2, 8, seed=9, pad_q=2)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)


def test_seq_lens_are_seeded_and_in_range():
    a = wl.seq_lens(64, 512, 32768, seed=wl.SEED_BASE + 4)
    b = wl.seq_lens(64, 512, 32768, seed=wl.SEED_BASE + 4)
    assert torch.equal(a, b) and a.dtype == torch.int32
    assert int(a.min()) >= 512 and int(a.max()) <= 32768
