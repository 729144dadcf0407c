"""The calls can be captured into a CUDA graph (torch.cuda.graph) and replayed:
every launch enqueues on the caller's stream and allocates nothing once its
buffers exist, and the launches' programmatic-dependent-launch edges are
captured with them.  A replay gives the bits of the same calls run eagerly,
also after the inputs change in place between replays."""
import pytest
import torch

import gpu_harness as H
from vocab_wide_logprob_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _case(seed):
    return H.with_contrast(wl.variant(wl.QWEN_G8, name=f"graph_{seed}", B=2, G=4, P=6, C=40,
                                      V=4099, eos_id=4098, reward_p=0.5, seed=seed))


@pytest.mark.parametrize("fused", [False, True], ids=["two_pass", "fused"])
def test_step_replays_in_a_cuda_graph(fused):
    n = H.g()
    w = _case(400)
    w2 = wl.variant(w, seed=w.seed + 7)
    logits = wl.make_logits_cpu(w).cuda()
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    R = torch.from_numpy(wl.make_rewards(w)).cuda()
    mask, lens = n.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(R, w.G)
    dl = torch.empty_like(logits)
    out = n.grpo_loss_fwd(logits, w.P, ids, lens, adv)
    state = {}

    def enqueue():
        n.grpo_mask(ids, w.P, w.C, w.eos_id, mask, lens)
        n.grpo_advantage(R, w.G, adv)
        if fused:
            state["o"] = n.grpo_loss_fwd_bwd(logits, w.P, ids, lens, adv, None, None, 0.2, 0.0,
                                             0.0, None, out, out["workspace"], dl)
        else:
            o = n.grpo_loss_fwd(logits, w.P, ids, lens, adv, None, None, 0.2, 0.0, 0.0, out,
                                out["workspace"])
            n.grpo_loss_bwd(logits, w.P, ids, lens, o["lse"], o["w"], None, dl)

    def snapshot():
        torch.cuda.synchronize()
        return {k: out[k].clone() for k in ("logp", "lse", "w", "loss")} | {"dl": dl.clone()}

    enqueue()
    eager = snapshot()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        enqueue()
    dl.zero_()
    graph.replay()
    got = snapshot()
    for k in eager:
        assert torch.equal(_bits(eager[k]), _bits(got[k])), k
    assert n.grpo_check_error(out["workspace"]) == 0

    # new inputs in place: the replay follows them
    ids.copy_(torch.from_numpy(wl.make_ids(w2)))
    R.copy_(torch.from_numpy(wl.make_rewards(w2)))
    logits.copy_(wl.make_logits_cpu(w2).cuda())
    graph.replay()
    got2 = snapshot()
    enqueue()
    eager2 = snapshot()
    for k in eager2:
        assert torch.equal(_bits(eager2[k]), _bits(got2[k])), k
    assert not torch.equal(_bits(eager2["dl"]), _bits(eager["dl"]))


@pytest.mark.parametrize("host_dl", [False, True], ids=["dev_dlogits", "host_dlogits"])
def test_host_logits_step_replays_in_a_cuda_graph(host_dl):
    """The host-logits call captured into a CUDA graph and replayed, with the
    gradient in device memory or written straight into pinned host memory."""
    n = H.g()
    w = _case(410)
    logits = wl.make_logits_cpu(w)
    host = logits.pin_memory()
    staging = torch.empty(logits.shape, dtype=logits.dtype, device="cuda")
    ids = torch.from_numpy(wl.make_ids(w)).cuda()
    R = torch.from_numpy(wl.make_rewards(w)).cuda()
    _, lens = n.grpo_mask(ids, w.P, w.C, w.eos_id)
    adv = n.grpo_advantage(R, w.G)
    ref = n.grpo_loss_fwd_bwd(logits.cuda(), w.P, ids, lens, adv, None, None, 0.2, 0.0)
    torch.cuda.synchronize()
    dl0 = torch.empty(logits.shape, dtype=logits.dtype).pin_memory() if host_dl else None
    out = n.grpo_loss_fwd_bwd_host(host, w.P, ids, lens, adv, None, None, 0.2, 0.0,
                                   staging=staging, dlogits=dl0)
    dl = out["dlogits"]
    assert dl.is_cuda != host_dl
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        n.grpo_loss_fwd_bwd_host(host, w.P, ids, lens, adv, None, None, 0.2, 0.0, 0.0, None,
                                 out, out["workspace"], dl, staging=staging)
    dl.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert n.grpo_check_error(out["workspace"]) == 0
    for k in ("logp", "lse", "w", "loss"):
        assert torch.equal(_bits(ref[k]), _bits(out[k])), k
    assert torch.equal(_bits(ref["dlogits"]).cpu(), _bits(dl).cpu())
