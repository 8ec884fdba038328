"""The decode parity suites run again with the tcgen05 engine selected.

The tensor-memory decode kernel (int8 / e4m3fn caches, head_dim 128 or 256)
must meet the same oracle comparisons, tolerances, edge cases and flags as the
mma.sync kernel: the sparse-candidate and paged sweeps, the softcap / window /
sink variants, the float8 caches and the numerical-eligibility fallback.  Shapes
the engine does not serve (head_dim 64, fp16 caches, prefill) run on the mma.sync
kernel either way.
"""
import pytest
import torch

from test_gpu_fallback import *  # noqa: F401,F403
from test_gpu_fp8 import *  # noqa: F401,F403
from test_gpu_parity import *  # noqa: F401,F403
from test_gpu_variants import *  # noqa: F401,F403

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tcgen05_engine():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int8_kv_cache_gb300 as K
    K.load()
    with K.engine(K.ENGINE_TCGEN05):
        assert K.decode_engine() == K.ENGINE_TCGEN05
        yield
