"""Host-side checks of the transfer pipeline that need no GPU."""
import pytest

from dsa_indexer_cross_gb300.pipeline import HostLayerPipeline


def test_pipeline_needs_at_least_one_device_set():
    # the set count is checked before anything touches a device
    with pytest.raises(ValueError, match="n_sets"):
        HostLayerPipeline(None, None, ["full"], [], "cpu", n_sets=0)
