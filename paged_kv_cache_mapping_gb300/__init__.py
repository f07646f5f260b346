"""Paged KV cache attention for GB300 (placeholder until the binding lands)."""
