"""The synthetic target model's logits on the GPU side (a workload stand-in,
not part of the method): an expanded tree node gets its own draft logits plus
the seeded N(0, 0.5^2) noise of its slot; a retained node that was never
expanded gets the seeded N(0, 1) logits of its slot."""
import torch


def target_logits_from_draft(draft_logits, tree_exp, noise, fresh, out):
    """draft_logits [B][E][V]; tree_exp [B][S] (expanded slot or -1);
    noise, fresh [B][S][V]; writes out [B][S][V]."""
    V = draft_logits.shape[-1]
    exp = tree_exp.long()
    idx = exp.clamp(min=0)[..., None].expand(-1, -1, V)
    gathered = torch.gather(draft_logits, 1, idx)
    out.copy_(torch.where((exp >= 0)[..., None], gathered + noise, fresh))
    return out
