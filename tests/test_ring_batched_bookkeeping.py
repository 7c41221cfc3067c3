"""Host bookkeeping of the batched ring steps (ring_attn_*(batch_shards=True)),
checked on the CPU: which key/value block every shard holds at each step, and
that the dK / dV partial sums, passed on one shard per step, end where their
blocks belong.  Uses only the driver's block rotation (torch, no kernels)."""
import torch

from long_context_attention_attn_gb300.ring import _held_blocks


def test_held_blocks_follow_the_ring_schedule():
    # "Context parallelism and ring attention", section "Ring attention": at
    # step t shard r holds block (r - t) mod R
    b, R, n = 2, 4, 3
    x = torch.arange(b * R * n, dtype=torch.int64).view(b, R * n)  # value = row * R*n + pos
    for t in range(R):
        h = _held_blocks(x, R, t)
        assert h.shape == (b * R, n)
        for bi in range(b):
            for r in range(R):
                j = (r - t) % R
                want = x[bi, j * n:(j + 1) * n]
                assert torch.equal(h[bi * R + r], want)


def test_partial_sums_end_at_their_blocks():
    # every step adds, at shard r, a contribution tagged (shard r, block held);
    # the sums are then passed on one shard; after R steps position j must
    # hold exactly the contributions of every shard to block j
    b, R, n = 1, 5, 2
    acc = torch.zeros(b, R * n, dtype=torch.int64)
    blocks = torch.arange(R).repeat_interleave(n).view(1, R * n)  # block id of each row
    for t in range(R):
        held = _held_blocks(blocks, R, t).view(b * R, n)  # the block id each shard holds
        a = acc.view(b * R, n)
        for r in range(R):
            assert torch.all(held[r] == (r - t) % R)
            a[r] += 10 ** (r + 1) * (held[r] + 1)  # shard r's contribution to its block
        acc = _held_blocks(acc, R, 1).view(b, R * n)
    for j in range(R):
        want = sum(10 ** (r + 1) * (j + 1) for r in range(R))
        assert torch.all(acc[0, j * n:(j + 1) * n] == want)
