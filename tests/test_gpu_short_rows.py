"""GPU parity for the selection's short-row path (a live span of at most 8192
columns on the 128-bit path is kept in registers from its one read to the
end) and for its boundary with the streaming path, against the oracle in all
three modes.  Each case is built to reach one branch of that path: the
boundary lengths, every tier of its row top-k (the K-th above -inf, inside the
-inf tier, below it), a -NaN block maximum (which sends the row to the
streaming path), starts, row_repeat, an edge column kept past the width, and
block sizes 4 to 128."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tests.gpu_util import Case
from tests.test_gpu_parity import check_all_modes  # noqa: F401  (the module's fixture builds the library)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

NEG_NAN = np.uint32(0xFFC00000).view(np.float32)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import sparse_attention_indexer_live_gb300 as dsa
    dsa.build()
    dsa.load()


def _rows(n, W, seed):
    return np.random.default_rng(seed).standard_normal((n, W)).astype(np.float32)


def test_lengths_around_the_register_path_limit():
    # 8192 columns is the largest span the short-row path takes; 8193 and
    # longer stream; the short ones straddle K and Kb * B
    W = 20000
    ends = [8191, 8192, 8193, 8196, 9000, 2047, 2048, 2049, 2056, 2057, 2100, 4096]
    x = _rows(len(ends), W, 1)
    check_all_modes(Case(x, None, ends, width=W, block_size=8, block_topk=256, row_topk=2048),
                    what="limit")


def test_row_topk_tiers():
    # L = 2100 > K = 2048 with 263 blocks > Kb = 256: 257 kept blocks (2056 columns)
    W, B, Kb, K = 4096, 8, 256, 2048
    x = _rows(4, W, 2)
    # row 0: the K-th is above -inf (plain case)
    # row 1: 40 kept columns hold -inf, so the K-th falls inside the -inf tier
    #        (the tier is cut by column rank)
    # row 2: kept columns hold -NaN values (never a whole block): the K-th is
    #        below -inf, among them
    # row 3: both
    for r in (1, 3):
        x[r, 8:2100:50] = -np.inf
    for r in (2, 3):
        x[r, 1:2100:7] = NEG_NAN
    check_all_modes(Case(x, None, [2100] * 4, width=W, block_size=B, block_topk=Kb, row_topk=K),
                    what="tiers")


def test_negative_nan_block_maximum_takes_the_streaming_path():
    W = 3000
    x = _rows(3, W, 3)
    x[0, 80:88] = NEG_NAN          # a whole block of -NaN: its maximum is -NaN
    x[1, 2992:3000] = NEG_NAN      # the last block
    x[2, 0:8] = NEG_NAN
    check_all_modes(Case(x, None, [2500, 3000, 700], width=W, block_size=8, block_topk=64,
                         row_topk=1000), what="-NaN block")


def test_starts_and_row_repeat():
    W = 10000
    x = _rows(6, W, 4)
    # aligned starts (the 128-bit path): [0, s) is masked; unaligned: streaming path
    case = Case(x, [0, 4, 64, 100, 3, 8], [5000, 2100, 6000, 9000, 4000, 8200], width=W,
                block_size=8, block_topk=128, row_topk=1024)
    check_all_modes(case, what="starts")
    y = _rows(8, W, 5)
    for causal in (True, False):
        case = Case(y, None, [3000, 2200, 9000, 500], width=W, block_size=8, block_topk=200,
                    row_topk=1500, row_repeat=2, causal=causal)
        check_all_modes(case, what=f"rep2 causal={causal}")


def test_edge_column_kept_past_the_width():
    # ends past W put the pin past the buffer: only column W - 1 of the edge is
    # kept; W = 4099 leaves a partial last vector, W = 4100 a whole one
    for W in (4099, 4100):
        x = _rows(4, W, 6)
        x[:, W - 1] = -5.0  # the edge column is kept however small it is
        case = Case(x, None, [W + 1, W + 9, W + 30, W], width=W, block_size=8, block_topk=64,
                    row_topk=600)
        check_all_modes(case, what=f"edge W={W}")


@pytest.mark.parametrize("B,Kb,K", [(4, 300, 1500), (16, 100, 1000), (32, 60, 1800), (64, 20, 1200),
                                    (128, 10, 1300)])
def test_block_sizes(B, Kb, K):
    W = 9000
    x = _rows(5, W, 7 + B)
    ends = [8192, 5000, 1300, 8000, 9000]
    check_all_modes(Case(x, None, ends, width=W, block_size=B, block_topk=Kb, row_topk=K),
                    what=f"B={B}")
