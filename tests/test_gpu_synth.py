"""The CUDA input generator gives the NumPy generator's bits."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("count,offset,std", [(1, 0, 1.0), (1000, 0, 1e-3), (70001, 12345, 0.02)])
def test_gpu_generator_matches_cpu_bits(dtype, count, offset, std):
    import torch
    from synth.gpu import fill_normal
    t = torch.empty(count, dtype=torch.float32 if dtype == "f32" else torch.bfloat16, device="cuda")
    fill_normal(t, 7, 99, np.float32(std), offset=offset)
    got = t.float().cpu().numpy()
    want = synth.normal(7, 99, (count,), std=np.float32(std), dtype=dtype, offset=offset)
    np.testing.assert_array_equal(got, want.astype(np.float32))
