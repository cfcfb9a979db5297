"""Seeded synthetic workloads shared by the tests, the benchmark and the oracle."""
from .gen import (WORKLOADS, Workload, fill, make_attn_inputs, make_grad_output, make_scorer_inputs,
                  plant_groups, plant_positions, small)

__all__ = ["WORKLOADS", "Workload", "fill", "make_attn_inputs", "make_grad_output", "make_scorer_inputs",
           "plant_groups", "plant_positions", "small"]
