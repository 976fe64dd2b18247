"""Vocabulary-sharded (tensor-parallel) phases, emulated on one GPU: W is cut
into R shards of whole 256-column tiles, each shard's partials are computed on
its own W slice, the blocks are stacked as an all-gather would deliver them, and
the sharded merge must give the unsharded bits for every R.  Both phases are
also checked against the fp64 oracle on their own: each shard's records
against the oracle's per-block statistics of the same global tiles (global
argmax indices), and the merged logp / lse / argmax against the oracle's
logprob, at the parity tolerances of the unsharded path."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bitwise, assert_block_records, assert_parity, to_dev
from invariant_token_logprob_gb300.inputs import lm_head_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import invariant_token_logprob_gb300 as rlk
    rlk.lib()


def _sharded(rlk, d, V, R, it=1.0):
    bn = rlk.vocab_tile()
    nvt = (V + bn - 1) // bn
    nvt_s = (nvt + R - 1) // R
    T = d["h"].shape[0]
    buf = torch.full((R, T, nvt_s, 4), float("nan"), device="cuda")
    for r in range(R):
        lo = r * nvt_s * bn
        hi = min((r + 1) * nvt_s * bn, V)
        if lo >= V:
            continue
        out = buf[r, :, : (hi - lo + bn - 1) // bn].contiguous()
        rlk.logprob_partials_shard(d["h"], d["W"][lo:hi].contiguous(), d["targets"], V, lo, it,
                                   out=out)
        buf[r, :, : out.shape[1]] = out
    rlk.check_device_error()
    return buf, nvt_s


@pytest.mark.parametrize("T,H,V", [(70, 256, 3000), (5, 512, 151936), (300, 128, 257),
                                   (4, 64, 250000)])  # rows of 977 tiles
def test_sharded_merge_equals_unsharded_for_every_shard_count(T, H, V):
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(T, H, V, seed=T))
    full = tuple(x.cpu().numpy() for x in rlk.logprob(d["h"], d["W"], d["targets"]))
    P = rlk.logprob_partials(d["h"], d["W"], d["targets"]).cpu().numpy()
    nvt = P.shape[1]
    for R in (1, 2, 3, 4, 7, 8):
        if (R - 1) * ((nvt + R - 1) // R) >= nvt:
            continue  # that R would leave a shard without tiles
        buf, nvt_s = _sharded(rlk, d, V, R)
        # each shard's records are the unsharded records of its tiles, bit for bit
        b = buf.cpu().numpy()
        for r in range(R):
            j0, j1 = r * nvt_s, min((r + 1) * nvt_s, nvt)
            assert np.array_equal(b[r, :, : j1 - j0].view(np.uint32), P[:, j0:j1].view(np.uint32))
        got = tuple(x.cpu().numpy() for x in rlk.lse_merge_sharded(buf, d["targets"], V))
        assert_bitwise(full, got, f"R={R}")


@pytest.mark.parametrize("T,H,V,R,it", [(70, 256, 3000, 3, 1.0), (5, 512, 151936, 4, 1.0),
                                         (300, 128, 1000, 2, float(np.float32(1 / 0.7))),
                                         (33, 192, 20000, 7, 1.0)])
def test_sharded_phases_match_oracle(olib, T, H, V, R, it):
    import invariant_token_logprob_gb300 as rlk
    d = lm_head_inputs(T, H, V, seed=100 + T)
    dd = to_dev(d)
    bn = rlk.vocab_tile()
    nvt = (V + bn - 1) // bn
    buf, nvt_s = _sharded(rlk, dd, V, R, it)
    b = buf.cpu().numpy()
    bs = oracle.block_stats(d["h"], d["W"], d["targets"], bn, it, lib=olib)
    for r in range(R):
        j0, j1 = r * nvt_s, min((r + 1) * nvt_s, nvt)
        if j0 >= nvt:
            continue
        assert_block_records(np.ascontiguousarray(b[r, :, : j1 - j0]), bs, d["h"], d["W"], bn,
                             it, j0=j0, what=f"shard {r} of {R}")
    got = tuple(x.cpu().numpy() for x in rlk.lse_merge_sharded(buf, dd["targets"], V))
    rlk.check_device_error()
    ref = oracle.logprob(d["h"], d["W"], d["targets"], it, lib=olib)
    assert_parity(got, ref, what=f"sharded merge R={R}")


def test_shard_boundaries_are_checked():
    import invariant_token_logprob_gb300 as rlk
    d = to_dev(lm_head_inputs(4, 64, 1000, seed=1))
    with pytest.raises(rlk.RlkError) as e:
        rlk.logprob_partials_shard(d["h"], d["W"][100:600].contiguous(), d["targets"], 1000, 100)
    assert e.value.status == 1
    with pytest.raises(rlk.RlkError) as e:  # a shard that ends mid-tile before V
        rlk.logprob_partials_shard(d["h"], d["W"][0:300].contiguous(), d["targets"], 1000, 0)
    assert e.value.status == 1
