"""Host logic of the Python binding, on CPU: cache descriptors, argument checks
before any call reaches the library, and the decode step's input arena (the
block of memory one host-to-device copy moves per step)."""

import pytest
import torch

import mla_absorbed_latent_02_gb300 as mla


def test_contiguous_cache_descriptor():
    c = mla.Cache.contiguous(3, 40, device="cpu")
    assert tuple(c.storage.shape) == (3, 40, 576) and c.storage.dtype == torch.bfloat16
    d = c.desc
    assert (d.paged, d.num_seqs, d.capacity, d.num_blocks, d.max_blocks) == (0, 3, 40, 0, 0)
    assert d.base == c.storage.data_ptr() and not d.block_table
    f = mla.Cache.contiguous(2, 8, device="cpu", fp8=True)
    assert tuple(f.storage.shape) == (2, 8, 656) and f.storage.dtype == torch.uint8 and f.fp8


def test_paged_cache_descriptor():
    bt = torch.tensor([[3, 1, -1], [0, 2, 4]], dtype=torch.int64)
    for fp8, row in ((False, 576), (True, 656)):
        c = mla.Cache.paged_pool(5, bt, device="cpu", fp8=fp8)
        assert c.storage.shape[-1] == row and tuple(c.storage.shape[:2]) == (5, 64)
        d = c.desc
        assert (d.paged, d.num_seqs, d.num_blocks, d.max_blocks) == (1, 2, 5, 3)
        assert c.block_table.dtype == torch.int32
        assert d.block_table == c.block_table.data_ptr()


def test_cache_rejects_bad_storage():
    with pytest.raises(ValueError):
        mla.Cache(torch.zeros(2, 4, 576, dtype=torch.float32), False, 2, 4)
    with pytest.raises(ValueError):
        mla.Cache(torch.zeros(2, 4, 512, dtype=torch.bfloat16), False, 2, 4)
    with pytest.raises(ValueError):
        mla.Cache(torch.zeros(2, 4, 576, dtype=torch.bfloat16), False, 2, 4, fp8=True)
    with pytest.raises(ValueError):   # paged without an int32 [B, max_blocks] table
        mla.Cache(torch.zeros(2, 64, 576, dtype=torch.bfloat16), True, 2, 0,
                  torch.zeros(4, dtype=torch.int32))


def test_pointer_checks_reject_host_memory():
    with pytest.raises(ValueError):
        mla._ptr(torch.zeros(4), torch.float32, "x")        # a host tensor never reaches a kernel
    with pytest.raises(ValueError):
        mla._out_ptr(torch.zeros(4, dtype=torch.bfloat16), torch.bfloat16, "out")   # not pinned
    assert mla._ptr(None) is None


class _FakeCtx:
    def alloc_workspace(self, H, B, Hq, device="cpu"):
        return torch.empty(16, dtype=torch.float32, device=device)


@pytest.mark.parametrize("B,Hq,H,n_new", [(64, 1, 16, None), (3, 2, 128, 5), (1, 64, 16, 64)])
def test_decode_step_input_arena(B, Hq, H, n_new):
    cache = mla.Cache.contiguous(B, 16, device="cpu")
    w = torch.zeros(H, 128, 512, dtype=torch.bfloat16)
    st = mla.DecodeStep(_FakeCtx(), cache, w, w, B, Hq, n_new=n_new)
    n = B * Hq if n_new is None else n_new
    want = {"c_kv": ((n, 512), torch.bfloat16), "k_rope": ((n, 64), torch.bfloat16),
            "seq_idx": ((n,), torch.int32), "pos": ((n,), torch.int32),
            "q_nope": ((B, Hq, H, 128), torch.bfloat16), "q_rope": ((B, Hq, H, 64), torch.bfloat16),
            "q_pos": ((B, Hq), torch.int32), "seq_lens": ((B,), torch.int32)}
    base = st._arena.data_ptr()
    spans = []
    for name, (shape, dt) in want.items():
        t = getattr(st, name)
        assert tuple(t.shape) == shape and t.dtype == dt, name
        off = t.data_ptr() - base
        assert off % 256 == 0, name                          # every input starts 256-byte aligned
        spans.append((off, off + t.numel() * t.element_size(), name))
    spans.sort()
    for (a0, a1, na), (b0, b1, nb) in zip(spans, spans[1:]):
        assert a1 <= b0, (na, nb)                            # disjoint
    assert spans[-1][1] <= st._arena.numel()
    assert st.input_bytes == sum(e - s for s, e, _ in spans)
    # writing a view writes the arena (the step copies the arena, not the views)
    st.seq_lens.fill_(7)
    assert torch.equal(st._arena[spans[[s[2] for s in spans].index("seq_lens")][0]:][:4].view(torch.int32),
                       torch.tensor([7], dtype=torch.int32))
