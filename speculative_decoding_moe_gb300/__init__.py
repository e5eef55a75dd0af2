"""GB300-native MoE block-verify for speculative decoding (libdfv.so + binding)."""
from . import inputs  # noqa: F401
