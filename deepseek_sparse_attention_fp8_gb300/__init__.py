"""GB300-native DeepSeek Sparse Attention step (sm_103a CUDA behind a C ABI).

Importing the package loads nothing; `deepseek_sparse_attention_fp8_gb300.api`
loads the CUDA library and fails loudly if it has not been built.
"""
