"""Seeded synthetic input generators shared by the tests and the benchmark."""
from .gen import *  # noqa: F401,F403
