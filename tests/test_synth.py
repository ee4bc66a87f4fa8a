"""The shared input generator: published test vectors and agreement of its two forms."""
import numpy as np
import torch

from video_vae_decoder_gb300 import synth


def test_splitmix64_published_sequence():
    # SplitMix64 started from state 0 (key 0): the widely published first outputs.
    out = synth.splitmix64_np(0, np.arange(3))
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_fnv1a64_vectors():
    assert synth.fnv1a64("") == 0xCBF29CE484222325
    assert synth.fnv1a64("a") == 0xAF63DC4C8601EC8C


def test_normals_look_normal():
    x = synth.standard_normal_at(0, "t/stat", np.arange(200_000))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    assert abs(np.mean(x ** 3)) < 0.03 and abs(np.mean(x ** 4) - 3) < 0.05


def test_counter_based_random_access():
    full = synth.normal_f32((1000,), 3, "t/ra", 0.5, 2.0)
    idx = np.array([0, 1, 17, 998, 999])
    some = (0.5 + 2.0 * synth.standard_normal_at(3, "t/ra", idx)).astype(np.float32)
    np.testing.assert_array_equal(full[idx], some)


def test_torch_form_matches_numpy_form():
    shape = (3, 5, 7, 16)
    a = synth.normal_f32(shape, 0, "t/torch", 0.25, 1.5)
    b = synth.normal_torch(shape, 0, "t/torch", 0.25, 1.5, chunk=97).numpy()
    np.testing.assert_array_equal(a, b)
    ab = synth.normal_bf16(shape, 0, "t/torch", 0.25, 1.5)
    bb = synth.normal_torch(shape, 0, "t/torch", 0.25, 1.5, dtype=torch.bfloat16)
    np.testing.assert_array_equal(ab, bb.view(torch.int16).numpy().view(np.uint16))
