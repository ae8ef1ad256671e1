"""MoE expert-parallel dispatch layout, dispatch and combine on one GB300.

Importing the package loads nothing native; ``combine_ep_layout_05_gb300.ep``
loads the CUDA library (and raises if it has not been built).
"""
__version__ = "0.1.0"
