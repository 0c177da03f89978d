"""CPU oracle of the decoder layer (test infrastructure only; see llama_layer.py)."""
from . import llama_layer  # noqa: F401
