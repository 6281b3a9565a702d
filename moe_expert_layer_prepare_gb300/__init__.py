"""GB300-native batched grouped-masked block-FP8 MoE expert forward.

The compute path lives in the CUDA library ``libmoe_prep.so`` (built from
``csrc/``); ``binding`` marshals PyTorch tensors into its C ABI.  Importing this
package does not load the library; the first call through ``binding`` does, and
raises if the library has not been built.
"""
__all__ = ["binding", "synthetic"]
