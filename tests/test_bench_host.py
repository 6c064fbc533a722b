"""Host-side arithmetic of the benchmark, checked against the oracle's
layout: the roofline's algorithmic bytes and the reported bits per element
must agree with what a packed cache stream actually holds, for every code
mode (no GPU needed)."""
import numpy as np
import pytest

import bench
from oracle import vqkv_oracle as vo
from vector_quantized_bit_gb300 import _lib, synth

MODES = sorted(vo.GEOMETRY)


def test_every_mode_is_known_everywhere():
    assert MODES == [0, 1, 2, 3, 4]
    assert synth.MODE_GEOMETRY == vo.GEOMETRY
    assert sorted(bench.BITS) == MODES
    assert [_lib.VQKV_MODE_VQ2, _lib.VQKV_MODE_VQ15, _lib.VQKV_MODE_VQ4, _lib.VQKV_MODE_VQ3,
            _lib.VQKV_MODE_VQ125] == [vo.MODE_VQ2, vo.MODE_VQ15, vo.MODE_VQ4, vo.MODE_VQ3, vo.MODE_VQ125]


@pytest.mark.parametrize("mode", MODES)
def test_bits_per_element_matches_the_layout(mode):
    assert bench.BITS[mode] == vo.bits_per_element(mode)
    T = vo.TILE_TOKENS[mode]
    assert vo.code_bytes(mode, 64 * T) * 8 == bench.BITS[mode] * 64 * T * 128


@pytest.mark.parametrize("mode", MODES)
def test_algorithmic_bytes_are_stream_bytes_plus_codebooks_q_and_o(mode):
    """Whole tiles: the index term equals the K and V stream bytes of every
    (sequence, KV head); the rest is the fp16 codebooks, q and O."""
    w = synth.WORKLOADS[1].with_mode(mode).scaled(B=3, Hq=16, Hkv=4)
    T = vo.TILE_TOKENS[mode]
    lens = np.array([5 * T, 17 * T, T], dtype=np.int64)
    E, dsub = vo.GEOMETRY[mode]
    streams = 2 * w.Hkv * sum(vo.code_bytes(mode, int(n)) for n in lens)
    codebooks = 2 * w.Hkv * E * dsub * 2
    q_and_o = 2 * w.B * w.Hq * 128 * 2
    assert bench.algorithmic_bytes(w, lens) == streams + codebooks + q_and_o


def test_headline_step_bytes():
    """The 196k-token Llama step reads 100,712,448 algorithmic bytes at 2 bit."""
    w = synth.WORKLOADS[1]
    assert w.mode == vo.MODE_VQ2 and (w.B, w.Hq, w.Hkv, w.seq_len) == (1, 32, 8, 196608)
    assert bench.algorithmic_bytes(w, np.array([w.seq_len])) == 100_712_448
