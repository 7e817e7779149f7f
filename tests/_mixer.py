"""Seeded models with the mixer bodies for the tests (inputs only: weights, mixer parameters)."""
import numpy as np

import oracle
import synth


def small_mixer_model(seed=12, n_layers=4, D=256, F=512, V=300, dims=None):
    """A 3 GDN + 1 FA stack at small width: GDN 2 key / 6 value heads of 128, FA 3 query / 1 KV heads
    of 256, n_mix 768; seeded weights and mixer parameters."""
    d = dims or oracle.MixerDims(nk=2, nv=6, nq=3, nkv=1)
    n_mix, qg, kv = d.nv * d.dv, 2 * d.nq * d.dh, d.nkv * d.dh
    layers, params = [], []
    for l in range(n_layers):
        fa = l % 4 == 3
        L = {"kind": oracle.LAYER_FA if fa else oracle.LAYER_GDN}
        shapes = {"w_in": (0, (qg if fa else d.gdn_in, D)), "w_out": (1, (D, n_mix)), "w_gate": (4, (F, D)),
                  "w_up": (5, (F, D)), "w_down": (6, (D, F))}
        if fa:
            shapes.update({"w_k": (2, (kv, D)), "w_v": (3, (kv, D))})
        for key, (slot, shp) in shapes.items():
            L[key] = oracle.q4k_pack(synth.normal(seed, 1000 * l + slot, shp, 0.02))
        layers.append(L)
        params.append(mixer_params(d, seed, l, fa))
    lm = oracle.q8_0_pack(synth.normal(seed, 900000, (V, D), 0.02))
    emb = synth.normal(seed, 900001, (V, D), 1.0)
    m = oracle.Model(D, F, V, d.gdn_in, qg, kv, n_mix, layers, lm, emb)
    return m, d, layers, params, lm, emb


def mixer_params(d, seed, l, fa):
    """Seeded mixer parameters of layer l (tensor ids 1000*l + 10..15)."""
    if fa:
        return oracle.MixerParams(q_norm_w=1.0 + 0.1 * synth.normal(seed, 1000 * l + 14, (d.dh,)),
                                  k_norm_w=1.0 + 0.1 * synth.normal(seed, 1000 * l + 15, (d.dh,)))
    u = synth.uniforms(seed, 1000 * l + 11, d.nv)
    return oracle.MixerParams(conv_w=0.5 * synth.normal(seed, 1000 * l + 10, (d.conv_dim, d.conv)),
                              a_log=np.log(1.0 + 15.0 * u),
                              dt_bias=synth.normal(seed, 1000 * l + 12, (d.nv,)),
                              norm_w=1.0 + 0.1 * synth.normal(seed, 1000 * l + 13, (d.dv,)))


