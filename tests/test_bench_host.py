"""Host-side checks of bench.py: every kernel source it hashes exists."""
import os

import bench


def test_kernel_source_lists_name_existing_files():
    csrc = os.path.join(bench.ROOT, "vocabulary_lm_cross_gb300", "csrc")
    for kernel, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.exists(os.path.join(csrc, n)), (kernel, n)
        assert len(bench.kernel_sources_sha(kernel)) == 64
