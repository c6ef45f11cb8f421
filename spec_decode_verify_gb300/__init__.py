"""Placeholder; the binding is added with the CUDA library."""
