"""skv_merge_parts on the host (no GPU): containers of consecutive layer ranges
of a cache, each encoded on its own (here by the oracle, standing in for one
GPU per range), merge into the container of the whole cache byte for byte;
malformed, reordered or incomplete parts are refused."""
import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def skv():
    import lossless_kv_cache_fixed_gb300 as P
    P.build()
    return P


def _model(O, spec, sigma, counts, L):
    return O.Model(spec.dtype, L, spec.H, spec.T, spec.D, spec.Tb, spec.G, sigma, counts=counts)


def _parts(O, spec, cuts, block_scale=False):
    """(whole container, [part containers], fingerprint) for layer cuts."""
    w = synth.make(spec)
    kv, mu, sig, cnt = synth.to_numpy(w)
    m = O.Model(spec.dtype, spec.L, spec.H, spec.T, spec.D, spec.Tb, spec.G, sig, counts=cnt,
                block_scale=block_scale)
    rc, whole = O.encode(m, kv, mu)
    assert rc == 0
    parts = []
    for l0, l1 in zip(cuts[:-1], cuts[1:]):
        mp = O.Model(spec.dtype, l1 - l0, spec.H, spec.T, spec.D, spec.Tb, spec.G, sig[l0:l1],
                     counts=cnt, block_scale=block_scale)
        rc, part = O.encode(mp, kv[l0:l1], mu[l0:l1])
        assert rc == 0
        parts.append(part)
    return whole, parts, O.model_hash(m)


def _params(P, spec, flags=0):
    # the merge reads no device data: the model pointers stay NULL
    return P.SkvParams(spec.dtype, spec.Tb, spec.G, flags, None, None, None), \
        P.SkvShape(spec.L, 2, spec.H, spec.T, spec.D)


@pytest.mark.parametrize("name,cuts", [
    ("tiny-bf16", [0, 1, 2]),
    ("qwen3-8b-e4m3", [0, 1, 3, 4]),
])
def test_merge_of_layer_ranges_is_the_whole_container(skv, oracle_mod, name, cuts):
    spec = synth.WORKLOADS[name]
    if spec.L != cuts[-1]:
        # a small cache of the same recipe: a ragged last token block, 4 lanes
        spec = spec.scaled(L=cuts[-1], H=2, T=300, D=64, Tb=128, G=4, calib_draws=2)
    whole, parts, fp = _parts(oracle_mod, spec, cuts)
    params, shape = _params(skv, spec)
    out = np.zeros(whole.size + 64, dtype=np.uint8)
    rc, nb = skv.skv_merge_parts(params, shape, fp, parts, out)
    assert rc == skv.SKV_OK, skv.skv_strerror(rc)
    assert nb == whole.size and np.array_equal(out[:nb], whole)


def test_merge_with_block_scales(skv, oracle_mod):
    spec = synth.WORKLOADS["qwen3-0.6b-bf16-drift"].scaled(L=3, H=2, T=300, Tb=128, G=4,
                                                           calib_draws=2)
    whole, parts, fp = _parts(oracle_mod, spec, [0, 2, 3], block_scale=True)
    params, shape = _params(skv, spec, skv.SKV_FLAG_BLOCK_SCALE)
    out = np.zeros(whole.size, dtype=np.uint8)
    rc, nb = skv.skv_merge_parts(params, shape, fp, parts, out)
    assert rc == skv.SKV_OK and np.array_equal(out[:nb], whole)


def test_merge_refuses_bad_parts(skv, oracle_mod):
    spec = synth.WORKLOADS["tiny-bf16"].scaled(L=3)
    whole, parts, fp = _parts(oracle_mod, spec, [0, 1, 3])
    params, shape = _params(skv, spec)
    out = np.zeros(whole.size, dtype=np.uint8)
    # missing a layer range, or too many layers
    assert skv.skv_merge_parts(params, shape, fp, parts[:1], out)[0] == skv.SKV_ERR_ARG
    assert skv.skv_merge_parts(params, shape, fp, parts + parts[:1], out)[0] == skv.SKV_ERR_CORRUPT
    # a part of another shape (its token count changed in the header)
    bad = parts[1].copy()
    bad[20] ^= 1
    assert skv.skv_merge_parts(params, shape, fp, [parts[0], bad], out)[0] == skv.SKV_ERR_CORRUPT
    # malformed offsets inside a part
    bad = parts[1].copy()
    nc = 2 * 2 * 2 * 1
    off = bad[64:64 + 8 * (nc + 1)].view(np.uint64)
    off[2] = off[3] + 4
    assert skv.skv_merge_parts(params, shape, fp, [parts[0], bad], out)[0] == skv.SKV_ERR_CORRUPT
    # truncated part, and an output that is too small
    assert skv.skv_merge_parts(params, shape, fp, [parts[0], parts[1][:-4]], out)[0] == \
        skv.SKV_ERR_CORRUPT
    small = np.zeros(whole.size - 1, dtype=np.uint8)
    assert skv.skv_merge_parts(params, shape, fp, parts, small)[0] == skv.SKV_ERR_CAPACITY
    # the parts in the right order still merge
    rc, nb = skv.skv_merge_parts(params, shape, fp, parts, out)
    assert rc == skv.SKV_OK and np.array_equal(out[:nb], whole)
