"""The delayed capacity input of the prefix scheduler ("DSpark：既要猜得连贯…", 设计: the
production scheduler reads a capacity estimate delayed by two steps): the table read at step t
is the one measured at step t - delay, from one fixed buffer.  Host-side (CPU tensors)."""
import torch

import semi_autoregressive_drafting_gb300 as ds


def test_two_step_delay():
    init = torch.full((5,), -1.0, dtype=torch.float64)
    ring = ds.CapacityRing(init, delay=2)
    addr = ring.table.data_ptr()
    seen = []
    for t in range(6):
        tab = ring.advance(torch.full((5,), float(t), dtype=torch.float64))
        assert tab.data_ptr() == addr  # one fixed buffer, e.g. for a captured graph
        seen.append(float(tab[0]))
    assert seen == [-1.0, -1.0, 0.0, 1.0, 2.0, 3.0]


def test_no_delay():
    ring = ds.CapacityRing(torch.zeros(3, dtype=torch.float64), delay=0)
    assert float(ring.advance(torch.full((3,), 7.0, dtype=torch.float64))[0]) == 7.0
