"""Data parallelism over tokens: the layer's one exchange between GPUs.

Every token row of the transformed linear is independent in the forward and
the backward; only the skew-parameter gradients are sums over tokens.  So a
data-parallel job gives each rank its own tokens, runs the whole layer on
them with replicated weights, permutations and skew parameters, and sums the
packed gradients dtheta_P and dtheta_R over ranks -- the distributed data
parallel training of the page "POET-X: Memory-efficient LLM Training by
Scaling Orthogonal Transformation" (gist.science summary, section 4).  The
packed gradients are b(b-1)/2 per block, half the bytes of the dense dQ
blocks they come from, so they are what goes over the wire.

The sum (not the mean) is taken: the library's gradients are sums over the
rank's tokens, so the summed result is the gradient of the whole batch.
"""
import torch
import torch.distributed as dist


def token_shard(T_global: int, world: int, rank: int) -> slice:
    """This rank's contiguous token rows of a global batch of T_global tokens:
    the first T_global % world ranks take one row more than the others."""
    if world < 1 or not 0 <= rank < world or T_global < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(T_global, world)
    start = rank * base + min(rank, extra)
    return slice(start, start + base + (1 if rank < extra else 0))


def allreduce_dtheta(dtheta_P: torch.Tensor, dtheta_R: torch.Tensor, group=None,
                     async_op: bool = False):
    """Sum both packed gradients over the ranks of `group`, in place (one
    all-reduce per side, on the current stream for NCCL).  With `async_op`
    returns the two work handles so the caller can overlap other work."""
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return [] if async_op else None
    works = [dist.all_reduce(dtheta_P, op=dist.ReduceOp.SUM, group=group, async_op=async_op),
             dist.all_reduce(dtheta_R, op=dist.ReduceOp.SUM, group=group, async_op=async_op)]
    return works if async_op else None


class GradientExchange:
    """The exchange of a multi-layer backward, overlapped with it: the packed
    gradients of a layer are all-reduced (asynchronously) as soon as that
    layer's backward has produced them, so that the exchange of layer L runs
    while the backward of layer L-1 computes -- DDP's overlap of communication
    with the backward, one bucket per layer.  ``wait`` ends the step: it waits
    for every exchange issued since the last ``wait``.

    Each layer must own its gradient buffers (the exchange reads and writes
    them in place until ``wait`` returns); with NCCL the collectives are
    ordered after the work already queued on the current stream."""

    def __init__(self, group=None):
        self.group = group
        self.works = []

    def layer_done(self, dtheta_P: torch.Tensor, dtheta_R: torch.Tensor):
        self.works.extend(allreduce_dtheta(dtheta_P, dtheta_R, group=self.group, async_op=True))

    def pending(self) -> int:
        return len(self.works)

    def wait(self):
        works, self.works = self.works, []
        for w in works:
            w.wait()


def backward_layers(layers, xs, dy, exchange=None):
    """Backward of a chain of transformed linears (``layers[i]`` maps xs[i]
    to xs[i + 1]; ``dy`` is the gradient of the last output): every layer's
    backward in reverse order, the gradient of a layer's input feeding the
    layer before it, each layer's packed gradients handed to ``exchange`` as
    soon as they exist.  Returns the gradient of the chain's input."""
    g = dy
    for lay, x in zip(reversed(layers), reversed(xs)):
        g, dtp, dtr = lay.backward(x, g)
        if exchange is not None:
            exchange.layer_done(dtp, dtr)
    return g


def max_over_ranks(value: float, group=None, device=None) -> float:
    """The largest of one float per rank (a job is as slow as its slowest rank)."""
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return float(value)
    if device is None:
        device = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
