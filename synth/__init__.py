"""Seeded synthetic inputs for parallel constrained decoding (PCD).

This package draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CPU oracle and the CUDA path read what it makes:

* model shapes (`model_config`) for the tiny reference decoder, the
  Qwen2.5-1.5B-shaped and the Qwen2.5-7B-shaped decoders;
* decoder weights (`make_weights`): every linear and embedding matrix drawn as
  N(0, 0.02) in a fixed tensor order, optionally rounded to bf16;
* requests (`make_request`): prefix token ids and the fields of a closed
  schema (scaffold tokens plus candidate label token paths).
"""
from .shapes import ModelConfig, model_config, CONFIG_MODEL
from .weights import make_weights, Weights, bf16_bits_to_f32, write_pcdw
from .requests import Field, Request, make_request, make_requests

__all__ = [
    "ModelConfig", "model_config", "CONFIG_MODEL",
    "make_weights", "Weights", "bf16_bits_to_f32", "write_pcdw",
    "Field", "Request", "make_request", "make_requests",
]
