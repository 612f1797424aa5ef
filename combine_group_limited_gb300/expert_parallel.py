"""Expert parallelism across the ranks of a process group.

"Expert Parallelism (Parallelisme d'experts)" (polydesk.ai), section "Le
principe de base": each rank holds whole experts, here a contiguous block of
E / world experts; section "Le pattern de communication all-to-all": Phase 1
(dispatch) sends every token to the ranks of its chosen experts, Phase 2
(combine) brings the expert outputs back to the token's rank, where they
are summed weighted by the router scores.

Tokens are data-parallel: rank s routes its own batch of T_s tokens.  One
exchange step per direction:

  1. local layout of the rank's own entries with the world's ranks as the
     logical ranks (ep_get_layout): its send buffer is grouped by
     destination rank, then expert, then local token -- the local dispatch
     writes it (ep_dispatch);
  2. count all-gather: every rank learns counts[s][e], the entries of source
     s for expert e, and from them the split sizes of the exchange;
  3. dispatch all-to-all-v: rank d receives, from each source s in turn,
     the rows of s for its experts (expert by expert);
  4. a row permutation turns [source][expert] into [expert][source], so
     that rank d's receive buffer is exactly rows rank_off[d] ..
     rank_off[d+1] of the single-GPU layout of the concatenated batch
     (sources in rank order): each expert's rows contiguous, in global
     token order;
  5. combine: the inverse permutation, the all-to-all-v back, and the
     rank's local weighted combine (ep_combine) in slot order.

The split sizes of an all-to-all-v are host integers, so step 2 reads the
gathered counts back to the host: the one synchronisation the exchange
needs (the hyper.ai Hybrid-EP story notes that sizing the receive buffers
needs one unless a fixed maximum is used).

The local steps are passed in as `ops` (layout, dispatch, combine and a row
permutation); `cuda_ops()` gives the library's kernels for CUDA tensors.
The exchange uses torch.distributed (NCCL on GPUs, gloo on CPU tensors).
"""
import numpy as np
import torch
import torch.distributed as dist


class LocalOps:
    """The rank-local steps the exchange calls.

    layout(idx [T, k] int32, E, experts_per_rank) -> dict with "pos" [T, k],
        "expert_count" [E], "rank_count" [R] (torch tensors on idx's device)
    dispatch(x [T, H], pos [T, k], rows) -> [rows, H] receive rows
    combine(y [rows, H], pos [T, k], w [T, k]) -> [T, H]
    permute(rows [n, H], target [n] int64) -> out [n, H] with out[target[i]] = rows[i]
    """

    def __init__(self, layout, dispatch, combine, permute):
        self.layout, self.dispatch, self.combine, self.permute = layout, dispatch, combine, permute


def cuda_ops():
    """The library's kernels as the local steps (CUDA tensors, bf16 rows)."""
    from . import _binding as ep

    def layout(idx, E, epr):
        lay = ep.ep_get_layout(idx, E, epr)
        return {"pos": lay.pos, "expert_count": lay.expert_count, "rank_count": lay.rank_count}

    def dispatch(x, pos, rows):
        recv = torch.empty((rows, x.shape[1]), dtype=x.dtype, device=x.device)
        return ep.ep_dispatch(x, pos, "bf16", recv=recv)

    def combine(y, pos, w):
        return ep.ep_combine(y, pos, w)

    def permute(rows, target):
        # a one-slot dispatch is a row scatter: out[target[i]] = rows[i]
        n = rows.shape[0]
        out = torch.empty_like(rows)
        if n:
            ep.ep_dispatch(rows, target.to(torch.int32).view(n, 1).to(rows.device), "bf16", recv=out)
        return out

    return LocalOps(layout, dispatch, combine, permute)


class ExpertParallel:
    """One rank's side of the expert-parallel exchange (see the module
    docstring).  Rank r of the group holds experts [r * epr, (r + 1) * epr),
    epr = num_experts / world."""

    def __init__(self, num_experts, ops, group=None):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if num_experts % self.world:
            raise ValueError("num_experts must be a multiple of the world size")
        self.E = num_experts
        self.epr = num_experts // self.world
        self.ops = ops

    # ---- the plan of one exchange
    def plan(self, topk_idx):
        """Local layout and the exchange's split sizes and permutation."""
        E, epr, W, me = self.E, self.epr, self.world, self.rank
        lay = self.ops.layout(topk_idx, E, epr)
        counts = lay["expert_count"].to(torch.int64).reshape(1, E)
        gathered = [torch.empty_like(counts) for _ in range(W)]
        dist.all_gather(gathered, counts, group=self.group)
        cnt = torch.cat(gathered).cpu().numpy()                  # [W][E]: the one host read-back
        mine = slice(me * epr, (me + 1) * epr)
        send_splits = [int(c) for c in lay["rank_count"].cpu().numpy()]
        recv_splits = [int(cnt[s, mine].sum()) for s in range(W)]
        # received order: source s, then expert e (of mine), then s's tokens;
        # wanted: expert e, then source s, then tokens
        mine_cnt = cnt[:, mine]                                   # [W][epr]
        exp_base = np.concatenate([[0], np.cumsum(mine_cnt.sum(axis=0))[:-1]])   # first row of each expert
        src_in_exp = np.cumsum(mine_cnt, axis=0) - mine_cnt      # rows of lower sources within the expert
        target = np.empty(int(mine_cnt.sum()), np.int64)
        i = 0
        for s in range(W):
            for j in range(epr):
                n = int(mine_cnt[s, j])
                target[i:i + n] = exp_base[j] + src_in_exp[s, j] + np.arange(n)
                i += n
        return {"layout": lay, "send_splits": send_splits, "recv_splits": recv_splits,
                "target": torch.from_numpy(target), "inverse": torch.from_numpy(np.argsort(target)),
                "counts": cnt}

    # ---- phase 1
    def dispatch(self, x, topk_idx, plan=None):
        """Rows of this rank's experts, in the single-GPU layout order of the
        concatenated batch.  Returns (rows, plan)."""
        plan = plan or self.plan(topk_idx)
        pos = plan["layout"]["pos"]
        send = self.ops.dispatch(x, pos, int(pos.numel()))
        recv = torch.empty((sum(plan["recv_splits"]), x.shape[1]), dtype=x.dtype, device=x.device)
        self._all_to_all(recv, send, plan["recv_splits"], plan["send_splits"])
        return self.ops.permute(recv, plan["target"]), plan

    # ---- phase 2
    def combine(self, y, topk_w, plan):
        """Expert outputs y (rows of this rank's experts, in dispatch order)
        back to their tokens' ranks, summed there weighted by topk_w."""
        back = self.ops.permute(y, plan["inverse"])                # [source][expert] order again
        pos = plan["layout"]["pos"]
        mine = torch.empty((int(pos.numel()), y.shape[1]), dtype=y.dtype, device=y.device)
        self._all_to_all(mine, back, plan["send_splits"], plan["recv_splits"])
        return self.ops.combine(mine, pos, topk_w)

    def _all_to_all(self, out, inp, out_splits, in_splits):
        # rows travel as bytes: one element per byte keeps every dtype exact
        ob = out.contiguous().view(out.shape[0], -1).view(torch.uint8)
        ib = inp.contiguous().view(inp.shape[0], -1).view(torch.uint8)
        dist.all_to_all_single(ob, ib, out_splits, in_splits, group=self.group)
        if ob.data_ptr() != out.data_ptr():
            out.view(torch.uint8).view(ob.shape).copy_(ob)
