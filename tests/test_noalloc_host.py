"""Host-side checks of the allocation-free entry point (no GPU needed).

* The Python wrapper refuses a values tensor that is not a contiguous CUDA
  tensor before anything reaches the library.
* A numpy mirror of the slice bookkeeping that spmv_csr_run_noalloc's two
  kernels follow (slices of 2,048 nonzeros; per slice the rows found by
  lower_bound, one "head" for a row that started earlier, at most one "tail"
  for a row that continues; the fix-up adds a tail and the heads of the
  slices its row covers) shows on random row lengths, runs of empty rows at
  slice boundaries and very long rows that every row is written exactly
  once, and that every head the fix-up reads was written.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
S = pytest.importorskip("sparse_matrix_vector_gb300")

CHUNK = 2048


class FakeCudaInt32:
    """Stands in for a contiguous int32 CUDA tensor on a CPU-only machine."""

    def __init__(self, n):
        self.n = n
        self.dtype = torch.int32
        self.is_cuda = True
        self.device = torch.device("cuda", 0)

    def is_contiguous(self):
        return True

    def numel(self):
        return self.n

    def data_ptr(self):
        raise AssertionError("the wrapper must refuse before taking pointers")


@pytest.mark.parametrize("values", [torch.zeros(8, dtype=torch.float32),
                                    torch.zeros(8, dtype=torch.float64)])
def test_wrapper_refuses_host_or_wrong_type_values(values):
    rp, ci = FakeCudaInt32(5), FakeCudaInt32(8)
    with pytest.raises(TypeError):
        S.spmv_csr_run_noalloc(4, 4, rp, ci, values, None, None)


def lower_bound(row_ptr, n, target):
    return int(np.searchsorted(row_ptr[: n + 1], target, side="left"))


def mirror(row_ptr):
    """Which slice writes each row of y (directly or via the fix-up), and
    the heads the fix-up reads; mirrors the kernels' index arithmetic."""
    n = len(row_ptr) - 1
    nnz = int(row_ptr[-1])
    n_slices = (nnz + CHUNK - 1) // CHUNK
    writes = np.zeros(n, np.int64)
    head_written = np.zeros(n_slices, bool)
    tail_row = np.full(n_slices, -1)
    for k in range(n_slices):
        lo, hi = k * CHUNK, min((k + 1) * CHUNK, nnz)
        rb = lower_bound(row_ptr, n, lo)
        re = n if k == n_slices - 1 else lower_bound(row_ptr, n, hi)
        if min(int(row_ptr[rb]), hi) - lo > 0:
            head_written[k] = True
        for r in range(rb, re):
            if row_ptr[r + 1] > hi:
                assert tail_row[k] == -1, "two tails in one slice"
                tail_row[k] = r
            else:
                writes[r] += 1
    for k in range(n_slices):
        r = tail_row[k]
        if r < 0:
            continue
        last = (int(row_ptr[r + 1]) - 1) // CHUNK
        assert last > k
        assert head_written[k + 1: last + 1].all(), f"fix-up of row {r} reads an unwritten head"
        writes[r] += 1
    return writes


def lengths_cases():
    rng = np.random.default_rng(11)
    yield rng.integers(0, 9, 4000)
    yield np.concatenate([[0, 0, 3], [300_001], [0] * 5, [CHUNK - 4], rng.integers(0, 9, 500),
                          [4096], [0] * 7])
    # runs of empty rows exactly at slice boundaries
    yield np.tile([CHUNK, 0, 0, 0], 6)
    yield np.concatenate([[CHUNK - 1], [0] * 3, [1], [0] * 4, [2 * CHUNK], [0] * 2])
    yield np.zeros(50, np.int64)
    yield rng.integers(0, 3 * CHUNK, 60)
    lens = rng.zipf(2.0, 20000)
    yield np.minimum(lens, 5000)


@pytest.mark.parametrize("lengths", list(lengths_cases()), ids=lambda a: f"n{len(a)}")
def test_slice_bookkeeping_writes_every_row_once(lengths):
    row_ptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    if row_ptr[-1] == 0:
        return   # the entry point clears y with one memset instead
    writes = mirror(row_ptr)
    assert np.array_equal(writes, np.ones(len(lengths), np.int64))
