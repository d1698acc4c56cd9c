"""The Python conveniences over torch tensors: layouts that the C calls cannot
describe (different shapes, strides, dtypes or devices among the tensors of
one call, non-2-D tensors, unpacked exchange rows) are refused with
ValueError before anything reaches the library, so these run without a GPU."""
import pytest
import torch

import tile_level_collective_gb300 as P


def t(rows=8, cols=16, dtype=torch.float32):
    return torch.zeros(rows, cols, dtype=dtype)


def test_window_ops_need_one_layout():
    good = [t() for _ in range(3)]
    for bad in ([t(), t(8, 17), t()],                       # shape
                [t(), t(dtype=torch.bfloat16), t()],      # dtype
                [t(), t(8, 32)[:, :16], t()]):            # row pitch
        with pytest.raises(ValueError):
            P.reduce_scatter(bad)
        with pytest.raises(ValueError):
            P.allgather(bad)
        with pytest.raises(ValueError):
            P.allreduce(bad)
        with pytest.raises(ValueError):
            P.broadcast(bad)
    with pytest.raises(ValueError):
        P.treduce(good, t(8, 17))                           # dst differs
    with pytest.raises(ValueError):
        P.treduce([torch.zeros(4, 4, 4)] * 2, torch.zeros(4, 4, 4))   # not 2-D
    with pytest.raises(ValueError):
        P.treduce([t().t(), t().t()], t().t())              # columns not contiguous


def test_exchanges_need_packed_rows():
    packed = [t() for _ in range(2)]
    strided = [t(8, 32)[:, :16] for _ in range(2)]
    counts = [torch.zeros(2, dtype=torch.int32) for _ in range(2)]
    with pytest.raises(ValueError):
        P.all_to_all(strided, packed)
    with pytest.raises(ValueError):
        P.all_to_all_v(packed, strided, counts, counts)
    with pytest.raises(ValueError):
        P.all_to_all_v_combine(packed, [t(), t(8, 8)], counts)
