"""Per-token vocabulary softmax divergences on GB300 (sm_103a).

Generalized Jensen-Shannon divergence, forward/reverse KL, entropy and
selected log-probabilities between language-model logits, with closed-form
backward, computed by hand-written CUDA kernels behind the C ABI of
``include/vpd.h``. ``binding`` mirrors the C entry points; ``ops`` gives
autograd functions; ``synth`` generates seeded synthetic inputs.

Submodules load lazily so that importing the package needs neither a GPU nor
the built library.
"""
import importlib

__all__ = ["binding", "ops", "synth", "build", "jsd", "kl_div", "entropy", "logprobs", "jsd_fwdbwd", "cross_entropy",
           "topk_forward_kl"]


def __getattr__(name):
    if name in ("binding", "ops", "synth", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    if name in ("jsd", "kl_div", "entropy", "logprobs", "jsd_fwdbwd", "cross_entropy", "topk_forward_kl"):
        return getattr(importlib.import_module(f"{__name__}.ops"), name)
    raise AttributeError(name)
