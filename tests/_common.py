"""Glue between the seeded inputs (csa_synth) and the oracle: format conversion only."""
import numpy as np
import torch

import csa_synth
from oracle import csa_oracle as O


def f64(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().float().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def oracle_layer(cfg: csa_synth.Config) -> O.Layer:
    return O.Layer(dtype=cfg.dtype, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi,
                   Di=cfg.Di, topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps, rollback=cfg.rollback)


def oracle_comp(c: csa_synth.Compressor) -> O.Compressor:
    return O.Compressor(wkv=f64(c.wkv), wgate=f64(c.wgate), ape=f64(c.ape), norm_w=f64(c.norm_w), d=c.d)


def oracle_state(cache: csa_synth.Cache) -> dict:
    return dict(pool=f64(cache.pool), ikeys=f64(cache.ikeys), window=f64(cache.window),
                front_a=f64(cache.front_attn), front_i=f64(cache.front_index),
                n_rows=cache.n_rows.numpy().astype(np.int64), pos=cache.pos.numpy().astype(np.int64))


def step_tuple(si: csa_synth.StepInputs):
    return (f64(si.x), f64(si.q), f64(si.kv), f64(si.iq), f64(si.iw))


def rel_err_rows(a, b):
    """max over leading rows of max|a-b| / max|b| along the last axis."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    num = np.abs(a - b).max(axis=-1)
    den = np.abs(b).max(axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max()) if num.size else 0.0
