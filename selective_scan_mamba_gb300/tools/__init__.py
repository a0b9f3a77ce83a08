"""Measurement helpers (not part of the scan library)."""
