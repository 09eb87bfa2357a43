"""Seeded synthetic inputs shared by the CPU oracle and the GPU path.

Nothing here computes any part of the resolve method: this package only
draws selection traces (:mod:`workloads.traces`) and host-pool records
(:mod:`workloads.records`) for the workloads listed in
:mod:`workloads.configs`.
"""
from .configs import ALL, BY_NAME, Workload  # noqa: F401
