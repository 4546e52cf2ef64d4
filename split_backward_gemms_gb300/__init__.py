"""GB300 (sm_103a) split-backward MLP stage: F, B and W passes and the 1F1B /
ZB-H1 / ZB-H2 one-GPU replay, after "Zero Bubble Pipeline Parallelism".

The compute path is the CUDA library ``libzb_gb300.so`` (C ABI in
``include/zb.h``); ``split_backward_gemms_gb300.zb`` binds it with the same
names and loads the library on import (``import split_backward_gemms_gb300.zb``).
"""
