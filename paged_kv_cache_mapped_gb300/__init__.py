"""Paged KV-cache decode attention for GB300 (placeholder until the CUDA binding lands)."""
