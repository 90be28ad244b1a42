"""Head-sharded FastOCR focal layers: a sequence's attention heads split over
several GPUs (tensor parallelism), whole GQA groups per GPU.

FastOCR (gist.science technical summary, "Focal-Guided Pruning", cross-layer
propagation) makes one selection per sequence, shared by every head of every
non-focal layer, from image scores summed over all query heads. With the
heads sharded, each GPU can only form the share of the scores that its own
heads contribute, so a focal layer needs one exchange: the shares
[B, N_img] fp32 are summed across the GPUs (an all-reduce) before the top-k.
Every GPU then selects from the same summed scores, so all of them get the
same selection, and non-focal layers need no exchange at all (each GPU
attends its own heads over that selection).

This module holds the host side: which heads a rank owns and the score
all-reduce. DecodeAttention(score_reduce=...) runs the focal layers as
fastocr_focal_scores -> score_reduce -> fastocr_select.
"""
from __future__ import annotations


def shard_heads(q_heads: int, kv_heads: int, rank: int, world: int):
    """Contiguous KV-head range [kv0, kv1) of `rank` and its query heads
    [q0, q1) = [kv0*g, kv1*g) (g = q_heads // kv_heads), so every query head
    stays with the KV head it reads. KV heads are dealt as evenly as possible
    (the first kv_heads % world ranks take one more); a rank may hold none
    only if world > kv_heads, which is rejected."""
    if q_heads % kv_heads:
        raise ValueError("q_heads must be a multiple of kv_heads")
    if not 0 <= rank < world or world > kv_heads:
        raise ValueError("need 0 <= rank < world <= kv_heads")
    g = q_heads // kv_heads
    base, extra = divmod(kv_heads, world)
    kv0 = rank * base + min(rank, extra)
    kv1 = kv0 + base + (1 if rank < extra else 0)
    return kv0 * g, kv1 * g, kv0, kv1


def score_all_reduce(group=None):
    """score_reduce callback for DecodeAttention: sums the score shares of all
    ranks of `group` in place (torch.distributed all-reduce, SUM). Every rank
    receives the same summed tensor, hence the same selection."""
    import torch.distributed as dist

    def reduce(sigma):
        dist.all_reduce(sigma, op=dist.ReduceOp.SUM, group=group)
    return reduce
