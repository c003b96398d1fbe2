"""The seeded generator: determinism, moments, planted structure (CPU only)."""
import numpy as np

from synth import cpu as gen
from synth import recipe


def test_normal_stream_is_deterministic_and_sliceable():
    k = gen.stream_key(0, 42)
    a = gen.normal_bf16_bits(k, 0, 5000)
    b = gen.normal_bf16_bits(k, 1234, 100)
    assert np.array_equal(a[1234:1334], b)
    assert not np.array_equal(a[:100], gen.normal_bf16_bits(gen.stream_key(0, 43), 0, 100))


def test_normal_moments():
    x = gen.bf16_bits_to_f32(gen.normal_bf16_bits(gen.stream_key(1, 2), 0, 1 << 20)).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 1e-2
    assert np.abs(x).max() <= 6.0


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.0078125 + 2 ** -8 + 2 ** -10, -2.5, 3.0e-3], dtype=np.float32)
    bits = gen.f32_to_bf16_bits(x)
    back = gen.bf16_bits_to_f32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0                 # halfway between 1 and 1+2^-7: ties to even (1.0)
    assert back[2] == np.float32(1.015625)  # above halfway rounds up
    assert back[3] == -2.5


def test_hot_blocks_avoid_sinks_and_window():
    for i in (1, 2, 3):
        w = recipe.workload(i)
        for r, blocks in enumerate(gen.hot_blocks(w)):
            N = w.lengths[r]
            for g in blocks:
                assert g * w.G >= w.A and (g + 1) * w.G <= N - w.n
    assert len(gen.hot_blocks(recipe.workload(1))[0]) == 8


def test_planted_keys():
    w = recipe.small(lengths=(700, 300), Hq=4, Hkv=2, dk=64, hot=("frac", 0.3), salt=9)
    u = gen.mean_query_dirs(w)
    hot = gen.hot_token_mask(w)
    base = gen.normal_bf16_bits(w.key(recipe.TID_K), 0, w.T * w.Hkv * w.dk).reshape(w.T, w.Hkv, w.dk)
    K = gen.gen_k(w, 0, w.T, u, hot)
    kb, kk = gen.bf16_bits_to_f32(base), gen.bf16_bits_to_f32(K)
    cu = w.cu_seqlens()
    for r in range(w.R):
        assert np.array_equal(kk[cu[r]:cu[r] + 4], kb[cu[r]:cu[r] + 4] * 4)
    idx = np.flatnonzero(hot)
    assert len(idx) > 0
    req = np.searchsorted(np.asarray(cu), idx, side="right") - 1
    diff = kk[idx] - kb[idx]
    np.testing.assert_allclose(diff, 2.0 * u[req], atol=0.07)
    cold = np.flatnonzero(hot == 0)
    cold = cold[np.isin(cold, [c + j for c in cu[:-1] for j in range(4)], invert=True)]
    assert np.array_equal(kk[cold], kb[cold])
    np.testing.assert_allclose(np.linalg.norm(u, axis=-1), 1.0, atol=1e-6)


def test_config_geometry():
    c = recipe.CONFIGS
    assert c[1].T == 4096 and c[2].T == 32768 and c[4].T == 4 * 131072 and c[5].T == 64 * 32768
    assert all(4096 <= L <= 131072 for L in c[3].lengths) and c[3].R == 16
    assert (c[4].Hq, c[4].Hkv, c[4].dk, c[4].G) == (16, 2, 256, 32)
    assert (c[5].Hq, c[5].Hkv, c[5].dk, c[5].hdim) == (16, 8, 256, 3840)
