"""Host-side logic that needs no GPU: the binding's flag composition, the seeded
input generators, and the library's sizing of the attention block."""
import numpy as np
import pytest

from laplacian_nystr_linear_gb300 import _lib, api
from laplacian_nystr_linear_gb300.inputs import WORKLOADS, block_inputs, make_inputs


def _p(**kw):
    base = dict(B=1, H=1, grid_h=14, grid_w=14, d=32, m=49, lam=32.0)
    base.update(kw)
    return api.Params(**base)


def test_flags_compose_the_header_bits():
    assert _p().flags == 0
    assert _p(norm=True).flags == _lib.LAPNYS_NORM
    assert _p(kernel="gauss").flags == _lib.LAPNYS_GAUSS
    assert _p(norm=True, norm_batch=True, kernel="gauss").flags == (
        _lib.LAPNYS_NORM | _lib.LAPNYS_NORM_BATCH | _lib.LAPNYS_GAUSS)
    with pytest.raises(ValueError):
        _ = _p(kernel="softmax").flags


@pytest.mark.parametrize("tied", [False, True])
def test_block_inputs_are_seeded_shaped_and_rounded(tied):
    a = block_inputs(3, 2, 16, 24, 2, 8, "bf16", tied)
    b = block_inputs(3, 2, 16, 24, 2, 8, "bf16", tied)
    S = 2 if tied else 3
    assert a["x"].shape == (2, 16, 24) and a["dy"].shape == (2, 16, 24)
    assert a["w_qkv"].shape == (24, S * 16) and a["b_qkv"].shape == (S * 16,)
    assert a["w_o"].shape == (16, 24) and a["b_o"].shape == (24,)
    for n in a:
        np.testing.assert_array_equal(a[n], b[n])
        assert a[n].dtype == np.float32
        assert not (a[n].view(np.uint32) & 0xFFFF).any()   # bf16 values: low 16 bits zero
    c = block_inputs(4, 2, 16, 24, 2, 8, "f32", tied, bias=False)
    assert c["b_qkv"] is None and c["b_o"] is None
    assert (c["x"].view(np.uint32) & 0xFFFF).any()


def test_workload_inputs_bf16_and_tied():
    w = WORKLOADS["tied64k"].scaled(B=1, H=1, grid_h=16, grid_w=16)
    inp = make_inputs(w)
    assert inp["k"] is inp["q"]
    assert not (inp["q"].view(np.uint32) & 0xFFFF).any()


@pytest.fixture(scope="module")
def lib():
    from laplacian_nystr_linear_gb300 import build as b
    b.build()
    return _lib.load()


def test_block_sizes_track_the_shapes(lib):
    def ctx(B, tied=0, dtype=1):
        return lib.lapnys_block_ctx_bytes(B, 1024, 256, 4, 64, 64, 8, tied, dtype, 0)

    def ws(B, tied=0, dtype=1):
        return lib.lapnys_block_workspace_bytes(B, 1024, 256, 4, 64, 64, 8, tied, dtype, 0)

    assert 0 < ctx(1) < ctx(2) < ctx(4)
    assert ctx(2, tied=1) < ctx(2)                 # no saved K
    assert ctx(2, dtype=1) < ctx(2, dtype=0)       # bf16 saves half the bytes of fp32
    assert ws(2) >= lib.lapnys_workspace_bytes(2, 4, 1024, 64, 64, 8, 0)
    # the saved Q, K, V and concatenated heads: four [B][H][N][d] tensors of bf16
    assert ctx(2) - lib.lapnys_ctx_bytes(2, 4, 1024, 64, 64, 8, 0) >= 4 * 2 * 4 * 1024 * 64 * 2


def test_outlier_counts_match_the_drawn_tokens():
    # the counts are those of the heavy-tailed rows make_inputs writes: on a small
    # copy of the high-resolution workload, the rows that differ from the plain
    # N(0, 1) draw of the same seed are exactly the counted ones
    from laplacian_nystr_linear_gb300.inputs import outlier_counts
    w = WORKLOADS["hires16k"].scaled(B=2, H=3, grid_h=16, grid_w=16)
    with_out = make_inputs(w)
    plain = make_inputs(w.scaled(outliers=False))
    changed = ((with_out["q"] != plain["q"]).any(-1).sum(-1)
               + (with_out["k"] != plain["k"]).any(-1).sum(-1))
    np.testing.assert_array_equal(outlier_counts(w), changed)
    assert outlier_counts(w).sum() > 0
    assert not outlier_counts(w.scaled(outliers=False)).any()


def test_top_outlier_slices_are_the_largest_counts():
    from laplacian_nystr_linear_gb300.inputs import outlier_counts
    from tests._parity import top_outlier_slices
    w = WORKLOADS["hires16k"]
    c = outlier_counts(w)
    top = top_outlier_slices(w, 6)
    assert len(top) == 6
    assert min(c[b, h] for b, h in top) >= max(c[b, h] for b in range(w.B) for h in range(w.H)
                                                 if (b, h) not in top)


def test_oracle_pool_matches_the_serial_oracle():
    from tests._oracle_pool import _check_matches_serial
    _check_matches_serial()
