"""gk: GPT-2 decoder-step kernels for one GB300 (sm_103a), behind the C ABI in include/gk.h.

Import `gpt_decoder_gb300.gk` for the binding (it loads libgk.so) and
`gpt_decoder_gb300.model` for the training-step driver.
"""
