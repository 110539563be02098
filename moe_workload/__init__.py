"""Seeded synthetic workloads for the sparse-MoE expert path (inputs only, no method arithmetic)."""
from .configs import (WORKLOADS, Workload, MoEShape, Q4, ExpertWeights, LayerInputs, make_layer, make_x,
                      make_decode_x, make_expert_weights, custom_workload, zipf_logit_bias)
from . import gen

__all__ = ["WORKLOADS", "Workload", "MoEShape", "Q4", "ExpertWeights", "LayerInputs", "make_layer", "make_x",
           "make_decode_x", "make_expert_weights", "custom_workload", "zipf_logit_bias", "gen"]
