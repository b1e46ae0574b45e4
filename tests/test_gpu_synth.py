"""The input generator's device fill equals its host regeneration bit for
bit, so the CUDA path and the oracle see the same history."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "mid", "sinks"])
def test_device_history_equals_host(name):
    w = synth.WORKLOADS[name]
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, dtype=torch.float32, device="cuda")
    V = torch.empty(shape, dtype=torch.float32, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    for s in sorted({0, w.n_slots - 1} | set(int(x) for x in rng.integers(0, w.n_slots, 4))):
        lo = int(rng.integers(0, w.slot_ctx))
        hi = min(w.slot_ctx, lo + 64)
        for which, buf in (("k", K), ("v", V)):
            got = buf[s, lo:hi].cpu().numpy()
            want = w.hist_rows(which, s, lo, hi)
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (name, which, s, lo)
