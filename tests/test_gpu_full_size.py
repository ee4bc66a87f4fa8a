"""Every output element at the full sizes of the decoder workloads against the fp64 oracle, run the
way the GPU runs them (the same chunks, the same carried caches):

  * the C=256 decoder stage: three causal ResBlocks on [1, 12, 176, 312, 256] as three 4-frame
    chunks carrying their six caches (binding.cpp, `Decoder::resnet`; `decode_video`: the history
    crosses passes in the cache);
  * the widest stage: two causal ResBlocks on [1, 4, 44, 78, 1024] with carried history, through
    the direct convs (the norm applied in their operand prologue at Cin = 1024, the last round of
    tile pairs split into halves of 128 channels) and through the Winograd F(2x2, 3x3) convs;
  * the causal convs alone at both sizes, with history, bias and residual;
  * the 256 -> 12 output head on [1, 16, 704, 1248, 256] (every one of its 168 M outputs; the
    oracle runs in bands of rows, each convolved with its one-row halo).

Criterion (conv / ResBlock / head): relative L2 <= 4e-3 and max |err| <= 2^-7 max |ref| over the
whole output; the first norm's cache (GroupNorm + SiLU of the input) within one bf16 ulp. Every
ResBlock invocation of the stages is held to it with the oracle's own input and caches; the stages
as the GPU chains them (each block fed by the GPU's previous block) are also compared with the
oracle's chain, with the max bound growing by one rounding step per block (check_chain).
The oracle runs on the host cores: these tests take minutes, most of it CPU time."""
import numpy as np
import pytest
import torch

import oracle
from util import MAX_ABS_FRAC, to_dev, f32_dev, bits, conv_close, cache2_close, ConvErr, ulp_report
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))
G = 32


def check_chain(got, ref, what):
    """got[k][chunk], ref[k][chunk]: block k's outputs of a chain of ResBlocks in which each side
    feeds every block with its own previous block's bf16 output. The two chains drift apart by
    rounding: where fp32 and fp64 accumulations fall on either side of a bf16 rounding boundary,
    a value differs by one step, every following conv spreads such steps over its output, and the
    residual connection carries them on. Block k (from 0) is held to relative L2 <= 4e-3 and
    max |err| <= (k + 1) 2^-7 max |ref|: one rounding step at the largest magnitude per block."""
    for k in range(len(got)):
        g, r = np.concatenate(got[k], 1), np.concatenate(ref[k], 1)
        err = ConvErr(f"{what} chained, block {k}", max_abs_frac=(k + 1) * MAX_ABS_FRAC)
        err.add(g, r)
        rel, mx = err.rel_and_max()
        print(f"{what} chained block {k}: rel L2 {rel:.3e}, max |err| {mx:.4g} (2^-7 max|ref| = "
              f"{err.maxref / 128:.4g}), ulps {ulp_report(g, r)}")
        err.check()


def run_block(wan, x_bits, p_dev, c1_bits, c2_bits, valid):
    """One wan_resblock call on host inputs; returns (out, cache1, cache2) as bf16 bits."""
    N, T, H, W, C = x_bits.shape
    zeros = np.zeros((N, 2, H, W, C), np.uint16)
    c1 = to_dev(zeros if c1_bits is None else c1_bits)
    c2 = to_dev(zeros if c2_bits is None else c2_bits)
    out = wan.wan_resblock(to_dev(x_bits), p_dev, c1, c2, valid, G, EPS)
    return bits(out), bits(c1), bits(c2)


def check_block(got, ref, what):
    """One block fed the oracle's own input and caches: the conv / ResBlock criterion, and the first
    norm's cache (GroupNorm + SiLU of the same input) within one bf16 ulp."""
    out, c1, c2 = got
    r_out, r1, r2 = ref
    rel, mx = conv_close(out, r_out, what)
    print(f"{what}: rel L2 {rel:.3e}, max |err| {mx:.4g}, ulps {ulp_report(out, r_out)['counts']}")
    assert int(oracle.ulp_distance_bf16(c1, r1).max()) <= 1, f"{what}: cache 1"
    cache2_close(c2, r2, f"{what}: cache 2")


def dev_params(p):
    return {k: (f32_dev(v) if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()}


def test_stage_c256_three_resblocks_in_chunks_matches_oracle(wan):
    shape = (1, 12, 176, 312, 256)
    N, T, H, W, C = shape
    x = synth.normal_torch(shape, 0, "stage4/x", device="cuda", dtype=torch.bfloat16)
    host_blocks = [synth.resblock_params(C, 0, f"stage4/block{i}") for i in range(3)]
    blocks = [dev_params(p) for p in host_blocks]
    caches = [(torch.zeros((N, 2, H, W, C), dtype=torch.bfloat16, device="cuda"),
               torch.zeros((N, 2, H, W, C), dtype=torch.bfloat16, device="cuda")) for _ in range(3)]
    chained = [[] for _ in range(3)]  # chained[block][chunk]: the GPU stage fed by itself
    for i, s in enumerate(range(0, T, 4)):
        h = x[:, s:s + 4].contiguous()
        for k, (blk, (c1, c2)) in enumerate(zip(blocks, caches)):
            h = wan.wan_resblock(h, blk, c1, c2, i > 0, G, EPS)
            chained[k].append(bits(h))
    assert wan.wan_device_status() == 0
    xh = bits(x)
    del x, caches
    torch.cuda.empty_cache()

    # The oracle stage, chunk by chunk; every block invocation is also run on the GPU with the
    # oracle's own input and caches (9 full-size ResBlocks under the ResBlock criterion).
    state = [(None, None)] * 3
    ref = [[] for _ in range(3)]
    for i, s in enumerate(range(0, T, 4)):
        h = np.ascontiguousarray(xh[:, s:s + 4])
        nxt = []
        for k, (p, (c1, c2)) in enumerate(zip(host_blocks, state)):
            got = run_block(wan, h, blocks[k], c1, c2, i > 0)
            h, c1, c2 = oracle.resblock(h, p, G, EPS, c1, c2)
            check_block(got, (h, c1, c2), f"C=256 chunk {i} block {k}")
            nxt.append((c1, c2))
            ref[k].append(h)
        state = nxt
    assert wan.wan_device_status() == 0
    check_chain(chained, ref, "C=256 stage")


def run_block_winograd(wan, x_bits, p_dev, us, c1_bits, c2_bits, valid):
    """One wan_resblock_winograd call on host inputs; returns (out, cache1, cache2) as bf16 bits."""
    c1, c2 = to_dev(c1_bits), to_dev(c2_bits)
    out = wan.wan_resblock_winograd(to_dev(x_bits), p_dev, us[0], us[1], c1, c2, valid, G, EPS)
    return bits(out), bits(c1), bits(c2)


def test_stage_c1024_two_resblocks_with_history_matches_oracle(wan):
    # Both GPU paths of the widest stage against one oracle run: the direct convs (norm in the
    # operand prologue) and the Winograd F(2x2, 3x3) convs (norm in the input transform).
    shape = (1, 4, 44, 78, 1024)
    N, T, H, W, C = shape
    xh = synth.normal_bf16(shape, 0, "stage5/x")
    host_blocks = [synth.resblock_params(C, 0, f"stage5/block{i}") for i in range(2)]
    blocks = [dev_params(p) for p in host_blocks]
    us = [(wan.wan_winograd_weights(b["w1"]), wan.wan_winograd_weights(b["w2"])) for b in blocks]
    # the history left by a previous chunk (activated values of each conv's input)
    hist = [(synth.normal_bf16((N, 2, H, W, C), 0, f"stage5/block{i}/c1", 0.1, 0.6),
             synth.normal_bf16((N, 2, H, W, C), 0, f"stage5/block{i}/c2", 0.1, 0.6)) for i in range(2)]
    chained, chained_w = [], []
    h = hw = xh
    for k, (c1, c2) in enumerate(hist):
        h, _, _ = run_block(wan, h, blocks[k], c1, c2, True)
        hw, _, _ = run_block_winograd(wan, hw, blocks[k], us[k], c1, c2, True)
        chained.append([h])
        chained_w.append([hw])
    r = xh
    ref = []
    for k, (p, (c1, c2)) in enumerate(zip(host_blocks, hist)):
        got = run_block(wan, r, blocks[k], c1, c2, True)
        got_w = run_block_winograd(wan, r, blocks[k], us[k], c1, c2, True)
        r, c1o, c2o = oracle.resblock(r, p, G, EPS, c1, c2)
        check_block(got, (r, c1o, c2o), f"C=1024 block {k}")
        check_block(got_w, (r, c1o, c2o), f"C=1024 Winograd block {k}")
        ref.append([r])
    assert wan.wan_device_status() == 0
    check_chain(chained, ref, "C=1024 stage")
    check_chain(chained_w, ref, "C=1024 Winograd stage")


@pytest.mark.parametrize("shape,Cout", [((1, 4, 176, 312, 256), 256), ((1, 4, 44, 78, 1024), 1024)])
def test_conv_full_size_every_element(wan, shape, Cout):
    # The causal conv alone (operands as stored), with a two-frame history, bias and residual.
    N, T, H, W, Cin = shape
    name = f"fullconv/{Cin}"
    a = synth.normal_bf16(shape, 0, f"{name}/a")
    w = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    b = synth.normal_bf16((Cout,), 0, f"{name}/b", 0.0, 0.01)
    r = synth.normal_bf16((N, T, H, W, Cout), 0, f"{name}/r")
    c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c")
    cout = torch.empty((N, 2, H, W, Cin), dtype=torch.bfloat16, device="cuda")
    y = wan.wan_causal_conv3d(to_dev(a), to_dev(w), to_dev(b), to_dev(r), to_dev(c), cout)
    got = bits(y)
    assert wan.wan_device_status() == 0
    f = oracle.bf16_to_f64
    conv_close(got, oracle.causal_conv3d_f64(f(a), f(w), f(b), f(r), f(c)), f"conv Cin={Cin} full size")
    assert np.array_equal(bits(cout), a[:, -2:])


def test_head_full_size_every_element(wan):
    # [1, 16, 704, 1248, 256] ~ N(0, 1) -> 12 channels, weights N(0, 1/(27*256)), zero history.
    shape = (1, 16, 704, 1248, 256)
    N, T, H, W, C = shape
    x = synth.normal_torch(shape, 0, "head/full/x", device="cuda", dtype=torch.bfloat16)
    w = synth.normal_bf16((12, 3, 3, 3, C), 0, "head/full/w", 0.0, float(np.sqrt(1.0 / (27 * C))))
    y = wan.wan_causal_conv3d(x, to_dev(w))
    got = bits(y)
    assert wan.wan_device_status() == 0
    xh = bits(x)
    del x, y
    torch.cuda.empty_cache()
    wf = oracle.bf16_to_f64(w)
    err = ConvErr("head 256->12 full size")
    band = 32
    for r0 in range(0, H, band):
        r1 = min(r0 + band, H)
        lo, hi = max(r0 - 1, 0), min(r1 + 1, H)
        ref = oracle.causal_conv3d_products_f64(oracle.bf16_to_f64(xh[:, :, lo:hi]), wf)
        err.add(got[:, :, r0:r1], ref[:, :, r0 - lo:r0 - lo + (r1 - r0)])
    assert err.count == N * T * H * W * 12
    err.check()
