"""Fused ONNX Conv (+ folded BatchNorm, bias, ReLU/ReLU6) for GB300 (sm_103a)."""
