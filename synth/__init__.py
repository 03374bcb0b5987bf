"""Seeded synthetic inputs (no attention arithmetic); shared by tests, bench and smoke."""
from .inputs import *  # noqa: F401,F403
from .inputs import WORKLOADS, make_workload, workload_lens  # noqa: F401
