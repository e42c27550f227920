"""Fp64 CPU oracle for the Focus hot path.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the benchmark's CPU-baseline leg, never by the product path.
"""
from .focus_ref import *  # noqa: F401,F403
