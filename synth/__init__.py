"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks."""
from .workloads import (  # noqa: F401
    RESOLUTIONS, Workload, chunk_bounds, config, grid_tiles, image_tokens,
    make_inputs, video_tokens,
)
