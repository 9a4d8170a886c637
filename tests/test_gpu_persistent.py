"""The same parity cases with the persistent step kernel (VSD_STEP_PERSISTENT).

The other modules run the default mode, one launch per GEMM and attention.
Here every cache the cases create is switched to the single persistent
launch before its first step; the cases and their tolerances are theirs.
"""
import pytest

from speculative_decoding_block_gb300 import binding as _B
from tests.gpu_helpers import gpu
from tests.test_gpu_draft import test_half_b_mixed_drafter_bench_workload  # noqa: F401
from tests.test_gpu_draft import test_tiny_anchor_export_and_draft, tiny  # noqa: F401
from tests.test_gpu_sampling import test_tiny_sampled_every_prefix  # noqa: F401
from tests.test_gpu_step import tiny_setup  # noqa: F401
from tests.test_gpu_step import test_tiny_batch_every_prefix_length, test_tiny_consecutive_steps_match_oracle  # noqa: F401
from tests.test_gpu_workloads import test_half_b_bf16_one_request_full  # noqa: F401
from tests.test_gpu_workloads import test_half_b_mixed_bench_workload_all_requests  # noqa: F401
from tests.test_gpu_workloads import test_seven_b_shape_one_layer_full  # noqa: F401

pytestmark = gpu


@pytest.fixture(autouse=True)
def persistent_mode(monkeypatch):
    create = _B.vsd_kv_create

    def create_persistent(*args, **kwargs):
        kv = create(*args, **kwargs)
        _B.vsd_kv_set_step_kernel(kv, _B.STEP_PERSISTENT)
        return kv

    monkeypatch.setattr(_B, "vsd_kv_create", create_persistent)
