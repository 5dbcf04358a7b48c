"""AdamW in float64 -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py for who may import it).

The fine-tuning step that follows the LoRA backward updates the shared adapter weights in place with
AdamW ("DeltaServe: Host-Agnostic Co-Serving of Inference and Fine-Tuning for LLMs", section 3.2 "Backward
subprocess": optimizer updates applied directly to the shared adapter weights; section 4.1: AdamW, learning
rate 1e-3, weight decay 0.01).  The pages name the optimizer but do not print it; this is AdamW with
decoupled weight decay and bias-corrected moments, written out step by step:

    m      <- beta1 * m + (1 - beta1) * g
    v      <- beta2 * v + (1 - beta2) * g * g
    theta  <- theta * (1 - lr * wd)                                 (decoupled weight decay)
    theta  <- theta - (lr / (1 - beta1^t)) * m / (sqrt(v) / sqrt(1 - beta2^t) + eps)

t is the 1-based step count.  Every array is float64; only the listed adapters' blocks change.
"""
import math

import numpy as np


def adamw_step(theta, g, m, v, *, lr, beta1, beta2, eps, weight_decay, step):
    """One AdamW step on whole arrays (float64 copies are returned: theta, m, v)."""
    theta = np.array(theta, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = np.array(m, dtype=np.float64)
    v = np.array(v, dtype=np.float64)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    theta = theta * (1.0 - lr * weight_decay)
    denom = np.sqrt(v) / math.sqrt(bc2) + eps
    theta = theta - (lr / bc1) * m / denom
    return theta, m, v


def adamw_pool(theta, g, m, v, offsets, ranks, width, adapters, **hp):
    """AdamW on the [r_a, width] blocks of the listed adapters of a pool-shaped array; other entries unchanged."""
    theta = np.array(theta, dtype=np.float64)
    m = np.array(m, dtype=np.float64)
    v = np.array(v, dtype=np.float64)
    for a in adapters:
        sl = slice(int(offsets[a]), int(offsets[a]) + int(ranks[a]) * width)
        theta[sl], m[sl], v[sl] = adamw_step(theta[sl], g[sl], m[sl], v[sl], **hp)
    return theta, m, v
