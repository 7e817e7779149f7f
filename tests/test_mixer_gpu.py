"""GPU parity of the decode with the mixer bodies ("Qwen3.6-27B on Apple M3 Pro", model
architecture list: Gated DeltaNet layers with their short conv and recurrent state, gated
full-attention layers with qk-norm, partial RoPE and a KV cache; "Mac Qwen3.6-27B Metal Q4_K perf
diagnosis", section 4: both run on the GPU inside the one-submission decode), through the C ABI,
against the oracle's MixerDecoder on the same seeded inputs.

The mixer steps run in f32 on the GPU and in f64 in the oracle; the state carries rounding from
token to token.  The bar on the logits is the f32 matmul bar (|err| <= 1e-5 * sum|w x| + 1e-6 per
logit, cosine >= 0.999999), teacher-forced: both sides are fed the oracle's token every step.
"""
import numpy as np
import pytest

import oracle
from _mixer import small_mixer_model
from _util import check_f32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fak():
    from q4_weight_quantized_block_gb300 import build
    build.build()
    import q4_weight_quantized_block_gb300 as m
    assert torch.cuda.is_available()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_context(fak, m, d, layers, params, lm, emb, D, F, V, mode=0, max_ctx=64):
    lg = []
    for L in layers:
        g = {"kind": fak.FAK_LAYER_FA if L["kind"] == oracle.LAYER_FA else fak.FAK_LAYER_GDN}
        for key, arr in L.items():
            if key != "kind":
                g[key] = dev(arr)
        lg.append(g)
    mix_layers = [{k: dev(v) for k, v in p.arrays.items()} for p in params]
    mixer = {"gdn_nk": d.nk, "gdn_nv": d.nv, "fa_nq": d.nq, "fa_nkv": d.nkv, "fa_rot": d.rot,
             "rope_theta": d.theta, "eps": d.eps, "max_ctx": max_ctx, "layers": mix_layers}
    n_mix = d.nv * d.dv
    return fak.DecodeContext(D, F, V, d.gdn_in, 2 * d.nq * d.dh, d.nkv * d.dh, n_mix, lg, dev(lm), dev(emb),
                             mode=mode, mixer=mixer)


def run_teacher_forced(fak, ctx, dec, V, n_tokens, tok=5, what=""):
    tin = torch.zeros(1, dtype=torch.int32, device="cuda")
    tout = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(V, device="cuda")
    worst = 0.0
    for step in range(n_tokens):
        tin.fill_(tok)
        ctx.step(tin, tout, logits)
        assert ctx.status() == 0
        rt, rl, ra, _ = dec.decode_token(tok)
        worst = max(worst, check_f32(logits.cpu().numpy(), rl, ra, "%s logits, position %d" % (what, step)))
        got = int(tout.item())
        if got != rt:
            gap = rl[rt] - rl[got]
            assert gap <= 1e-5 * (ra[rt] + ra[got]) + 2e-6, (step, got, rt, gap)
        tok = rt
    return worst


SMALL = dict(D=256, F=512, V=300)


def test_mixer_decode_small_matches_oracle(fak):
    m, d, layers, params, lm, emb = small_mixer_model(seed=12, **SMALL)
    ctx = gpu_context(fak, m, d, layers, params, lm, emb, **SMALL)
    dec = oracle.MixerDecoder(m, d, params, max_ctx=64)
    run_teacher_forced(fak, ctx, dec, SMALL["V"], 12, what="small mixer stack")
    ctx.close()
    dec.close()


def test_mixer_decode_eight_layers_two_periods(fak):
    # two 4-layer periods: the state of every layer kind is carried by more than one layer
    m, d, layers, params, lm, emb = small_mixer_model(seed=13, n_layers=8, **SMALL)
    ctx = gpu_context(fak, m, d, layers, params, lm, emb, **SMALL)
    dec = oracle.MixerDecoder(m, d, params, max_ctx=64)
    run_teacher_forced(fak, ctx, dec, SMALL["V"], 8, tok=17, what="8-layer mixer stack")
    ctx.close()
    dec.close()


def test_mixer_decode_long_context(fak):
    # 1100 positions: rotary angles up to 1100 rad (reduced modulo 2 pi on the GPU), key and value
    # passes over more than a thousand cached rows (many full unrolled batches and a remainder)
    m, d, layers, params, lm, emb = small_mixer_model(seed=17, **SMALL)
    ctx = gpu_context(fak, m, d, layers, params, lm, emb, max_ctx=1200, **SMALL)
    dec = oracle.MixerDecoder(m, d, params, max_ctx=1200)
    tin = torch.zeros(1, dtype=torch.int32, device="cuda")
    tout = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(SMALL["V"], device="cuda")
    tok = 7
    for step in range(1100):
        tin.fill_(tok)
        ctx.step(tin, tout, logits)
        rt, rl, ra, _ = dec.decode_token(tok)
        if step % 50 == 0 or step >= 1090:
            assert ctx.status() == 0
            check_f32(logits.cpu().numpy(), rl, ra, "long context, position %d" % step)
        tok = rt
    assert ctx.status() == 0
    ctx.close()
    dec.close()


def test_mixer_one_launch_equals_per_matmul_and_reset(fak):
    m, d, layers, params, lm, emb = small_mixer_model(seed=14, **SMALL)
    one = gpu_context(fak, m, d, layers, params, lm, emb, mode=0, **SMALL)
    per = gpu_context(fak, m, d, layers, params, lm, emb, mode=1, **SMALL)
    assert one.launches_per_step() == 1 and per.launches_per_step() == 1 + 5 * 4 + 2
    tin = torch.zeros(1, dtype=torch.int32, device="cuda")
    ta, tb = torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
    la, lb = torch.empty(SMALL["V"], device="cuda"), torch.empty(SMALL["V"], device="cuda")
    first = None
    for t in (3, 1, 4, 1, 5, 9):
        tin.fill_(t)
        one.step(tin, ta, la)
        per.step(tin, tb, lb)
        assert one.status() == 0 and per.status() == 0
        a, b = la.cpu().numpy(), lb.cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "one launch != per matmul"
        if first is None:
            first = a.copy()
    # a new sequence: the same first token gives the first step's logits again, bit for bit
    one.reset()
    tin.fill_(3)
    one.step(tin, ta, la)
    assert one.status() == 0
    assert np.array_equal(la.cpu().numpy().view(np.uint32), first.view(np.uint32))
    one.close()
    per.close()


def test_mixer_decode_full_width_matches_oracle(fak):
    # the 27B widths (d_model 5120, SwiGLU 17408, GDN 16 key / 48 value heads, FA 24 / 4 heads, n_mix
    # 6144) over one 4-layer period (3 GDN + 1 FA) with a 16384-token head
    full = dict(D=5120, F=17408, V=16384)
    dims = oracle.MixerDims()
    m, d, layers, params, lm, emb = small_mixer_model(seed=15, dims=dims, **full)
    ctx = gpu_context(fak, m, d, layers, params, lm, emb, **full)
    dec = oracle.MixerDecoder(m, d, params, max_ctx=64)
    run_teacher_forced(fak, ctx, dec, full["V"], 4, tok=11, what="full-width mixer stack")
    ctx.close()
    dec.close()


def test_mixer_step_past_max_ctx_reports_and_recovers(fak):
    # max_ctx = 4: the fifth position has no cache row.  The step records FAK_ERR_DEVICE without
    # waiting out the readers' timeout, reading the status clears the state, and the next step is
    # position 0 of a new sequence again (bit for bit the first step's logits).
    import time
    m, d, layers, params, lm, emb = small_mixer_model(seed=18, **SMALL)
    ctx = gpu_context(fak, m, d, layers, params, lm, emb, max_ctx=4, **SMALL)
    tin = torch.full((1,), 3, dtype=torch.int32, device="cuda")
    tout = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(SMALL["V"], device="cuda")
    first = None
    for step in range(4):
        ctx.step(tin, tout, logits)
        assert ctx.status() == 0
        if first is None:
            first = logits.cpu().numpy().copy()
    t0 = time.time()
    ctx.step(tin, tout, logits)
    st = ctx.status()
    assert st == 7, st  # FAK_ERR_DEVICE
    assert time.time() - t0 < 0.5
    ctx.step(tin, tout, logits)
    assert ctx.status() == 0
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), first.view(np.uint32))
    ctx.close()


def test_mixer_rejects_bad_shapes(fak):
    m, d, layers, params, lm, emb = small_mixer_model(seed=16, **SMALL)
    with pytest.raises(fak.FakError) as ei:
        gpu_context(fak, m, d, layers, params, lm, emb, max_ctx=100000, **SMALL)
    assert ei.value.status == 2
