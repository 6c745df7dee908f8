"""idx_top1 (one-launch top-1 of each row of logits) against the oracle, through
the C ABI: index bit-exact (ties to the lowest index, NaN read as -1e30), value,
the draft token column and position writes, and the per-row state left zero."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import sparse_attention_indexer_launch_gb300 as lib
    return lib


def _logits(seed, R, V):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, V)).astype(np.float32) * 4
    if R > 1:
        x[1] = rng.integers(-3, 4, V).astype(np.float32)           # heavy ties
    if R > 2:
        x[2, rng.integers(0, V, 50)] = np.nan                       # NaNs among normal values
    if R > 3:
        x[3] = np.nan                                                # all NaN -> index 0
    if R > 4:
        x[4] = -np.inf
        x[4, V // 2] = np.nan                                        # NaN (-1e30) beats -inf
    if R > 5:
        x[5] = 0.0
        x[5, ::3] = -0.0                                             # signed zeros tie
    if R > 6:
        j = rng.integers(0, V, 3)
        x[6, j] = np.float32(1e6)                                    # a tied maximum in different splits
    return x


def _run(lib, x, **kw):
    R, V = x.shape
    dx = torch.from_numpy(x).cuda()
    idx = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    val = torch.empty(R, dtype=torch.float32, device="cuda")
    state = torch.zeros(lib.top1_state_size(R), dtype=torch.uint8, device="cuda")
    lib.idx_top1(dx, idx, state, out_val=val, **kw)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), state


@pytest.mark.parametrize("R,V", [(1, 1), (3, 5), (8, 1000), (8, 151552), (7, 1_000_003), (40, 4099)])
def test_top1_matches_oracle(lib, orc, R, V):
    x = _logits(R * 1000 + V, R, V)
    idx, val, state = _run(lib, x)
    ref_idx, ref_val = orc.top1(x)
    assert np.array_equal(idx, ref_idx), (idx, ref_idx)
    assert np.array_equal(val.view(np.uint32), ref_val.view(np.uint32)) or np.array_equal(val, ref_val)
    assert int(state.count_nonzero()) == 0


def test_top1_unaligned_rows_and_two_calls(lib, orc):
    R, V, ld = 6, 20001, 20011
    base = torch.from_numpy(_logits(5, R, ld)).cuda()
    view = base[:, 1:1 + V]                          # 4-byte aligned only: scalar loads
    state = torch.zeros(lib.top1_state_size(R), dtype=torch.uint8, device="cuda")
    for _ in range(2):                               # the state is reused as the call leaves it
        idx = torch.empty(R, dtype=torch.int32, device="cuda")
        lib.idx_top1(view, idx, state, V=V)
        torch.cuda.synchronize()
        ref_idx, _ = orc.top1(view.cpu().numpy())
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert int(state.count_nonzero()) == 0


def test_top1_writes_draft_column_and_position(lib, orc):
    R, V = 5, 30000
    x = _logits(9, R, V)
    tokens = torch.full((R, 4), -1, dtype=torch.int32, device="cuda")
    positions = torch.arange(R, dtype=torch.int32, device="cuda") * 10
    idx, _, _ = _run(lib, x, tokens=tokens, token_col=2, positions=positions)
    ref_idx, _ = orc.top1(x)
    t = tokens.cpu().numpy()
    assert np.array_equal(t[:, 2], ref_idx) and (t[:, [0, 1, 3]] == -1).all()
    assert np.array_equal(positions.cpu().numpy(), np.arange(R) * 10 + 1)
