"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle."""
from .synth import (NAMES, LayerInputs, Workload, bf16_bits, bf16_to_f32, bf16_to_f64, key_head_scale,
                    layer_inputs, layer_inputs_device, named, random_tree, tree_parents)

__all__ = ["NAMES", "LayerInputs", "Workload", "bf16_bits", "bf16_to_f32", "bf16_to_f64", "key_head_scale",
           "layer_inputs", "layer_inputs_device", "named", "random_tree", "tree_parents"]
