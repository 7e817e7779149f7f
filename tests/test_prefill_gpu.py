"""GPU parity of the one-submission prefill forward (fak_prefill_*): P prompt tokens through the
stack as one CUDA graph, the projections-only floor of the pages' prefill ladder ("Qwen3.6-27B
GDN-hybrid Metal prefill -- isolation split", rung 3; "Mac Qwen3.6-27B Metal Q4_K perf diagnosis",
section 4: the resident prefill forward in one command buffer), against the oracle's
prefill_forward on the same seeded inputs, through the C ABI.

Every matmul is the bf16 tensor-core GEMM, whose bar is |err| <= 5e-3 * sum|w x| + 1e-5 per output
with cosine >= 0.9999.  Through the stack the two sides round their (slightly different)
activations to bf16 independently, so the checks are: every token's final hidden state within
cosine 0.9999 of the oracle's (the GEMM's cosine bar), the last token's logits within the GEMM bar
on the lm_head (the oracle's sum |w x|) and cosine >= 0.9999, and the token equal (or a near-tie
within that bar).
"""
import numpy as np
import pytest

import oracle
import synth
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


def stack(fak, seed, n_layers, D, F, V, GI, QG, KV, NM):
    lo, lg = [], []
    for l in range(n_layers):
        fa = l % 4 == 3
        Lo = {"kind": oracle.LAYER_FA if fa else oracle.LAYER_GDN}
        Lg = {"kind": fak.FAK_LAYER_FA if fa else fak.FAK_LAYER_GDN}
        shapes = {"w_in": (0, (QG if fa else GI, D)), "w_out": (1, (D, NM)), "w_gate": (4, (F, D)),
                  "w_up": (5, (F, D)), "w_down": (6, (D, F))}
        if fa:
            shapes.update({"w_k": (2, (KV, D)), "w_v": (3, (KV, D))})
        for key, (slot, shp) in shapes.items():
            o = oracle.q4k_pack(synth.normal(seed, 1000 * l + slot, shp, 0.02))
            Lo[key], Lg[key] = o, dev(o)
        lo.append(Lo)
        lg.append(Lg)
    lm = oracle.q8_0_pack(synth.normal(seed, 900000, (V, D), 0.02))
    emb = synth.normal(seed, 900001, (V, D), 1.0)
    om = oracle.Model(D, F, V, GI, QG, KV, NM, lo, lm, emb)
    return om, lg, dev(lm), dev(emb)


def run_case(fak, seed, n_layers, P, D, F, V, GI, QG, KV, NM):
    om, lg, lm, emb = stack(fak, seed, n_layers, D, F, V, GI, QG, KV, NM)
    toks = (np.arange(P) * 7919 + seed) % V
    ctx = fak.PrefillContext(D, F, V, GI, QG, KV, NM, lg, lm, emb, P)
    assert ctx.kernels() >= 1 + 7 * n_layers
    td = dev(toks.astype(np.int32))
    tout = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty(V, device="cuda")
    ctx.run(td, tout, logits)
    assert ctx.status() == 0
    h = torch.empty(P * D, device="cuda")
    ctx.read_hidden(h)
    torch.cuda.synchronize()
    rt, rl, ra, rh = om.prefill_forward(toks)
    hg = h.cpu().numpy().reshape(P, D).astype(np.float64)
    for p in range(P):
        cos = float(hg[p] @ rh[p] / np.linalg.norm(hg[p]) / np.linalg.norm(rh[p]))
        assert cos >= 0.9999, (p, cos)
    check_f32(logits.cpu().numpy(), rl, ra, "prefill logits", rel=5e-3, abs_=1e-5, cos_min=0.9999)
    got = int(tout.item())
    if got != rt:
        assert rl[rt] - rl[got] <= 5e-3 * (ra[rt] + ra[got]) + 2e-5, (got, rt)
    # a second run with the same tokens replays the same graph: bit for bit the same logits
    l1 = logits.clone()
    ctx.run(td, tout, logits)
    assert ctx.status() == 0
    assert torch.equal(l1.view(torch.int32), logits.view(torch.int32))
    ctx.close()


def test_prefill_small_stack(fak):
    # 4 layers (3 GDN + 1 FA) at small width; P spans two 256-token tiles and a ragged tail
    run_case(fak, 70, 4, 300, D=256, F=512, V=1000, GI=640, QG=512, KV=256, NM=256)


def test_prefill_single_token(fak):
    # P = 1: every GEMM has one token in its only token tile
    run_case(fak, 73, 4, 1, D=256, F=512, V=1000, GI=640, QG=512, KV=256, NM=256)


def test_prefill_gdn_in_not_a_multiple_of_128(fak):
    # the 27B GDN in_proj has 16480 rows: its last GEMM row tile is partial
    run_case(fak, 71, 4, 64, D=512, F=1024, V=512, GI=16480, QG=1024, KV=256, NM=512)


def test_prefill_full_width_one_period(fak):
    # the 27B widths over one 4-layer period at P = 32
    run_case(fak, 72, 4, 32, D=5120, F=17408, V=4096, GI=16480, QG=12288, KV=1024, NM=6144)
