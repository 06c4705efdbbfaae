"""libmoedc: MoE expert-parallel layout, dispatch and combine on one GB300.

The compute runs in the CUDA library libmoedc.so (built by build.build());
this package holds its ctypes binding (moedc) and the seeded synthetic
workloads (synth).
"""
from .moedc import (BF16, FP8_E4M3, SCALES_COL_MAJOR, SCALES_PER_TOKEN, Layout, MoedcError, alloc_recv, combine,
                    combine_e4m3, dequant_e4m3, moedc_combine_e4m3,
                    dispatch, layout, layout_dispatch, layout_workspace, load, moedc_combine,
                    moedc_dequant_e4m3, moedc_dispatch, moedc_layout, moedc_layout_dispatch,
                    moedc_layout_static_scratch, moedc_layout_workspace_bytes,
                    moedc_layout_dispatch_workspace_bytes, layout_dispatch_workspace,
                    moedc_rank_combine, moedc_rank_dispatch, moedc_rank_layout, rank_combine,
                    rank_dispatch, rank_layout, strerror)

__all__ = ["BF16", "FP8_E4M3", "SCALES_COL_MAJOR", "SCALES_PER_TOKEN", "Layout", "MoedcError", "alloc_recv",
           "combine", "combine_e4m3", "dequant_e4m3", "moedc_combine_e4m3",
           "dispatch", "layout", "layout_dispatch", "layout_workspace", "load", "moedc_combine",
           "moedc_dequant_e4m3", "moedc_dispatch", "moedc_layout", "moedc_layout_dispatch",
           "moedc_layout_static_scratch", "moedc_layout_workspace_bytes",
           "moedc_layout_dispatch_workspace_bytes", "layout_dispatch_workspace", "moedc_rank_combine",
           "moedc_rank_dispatch", "moedc_rank_layout", "rank_combine", "rank_dispatch",
           "rank_layout", "strerror"]
