"""RMSNorm (and LayerNorm) forward and backward for one GB300 (sm_103a).

The compute path is the C-ABI library ``librmsnorm.so`` built from ``csrc/``
(declared in ``include/rmsnorm.h``, ``include/layernorm.h`` and
``include/rmsnorm_double_backward.h``); ``binding`` is its thin Python front end
and ``autograd`` its PyTorch integration (``rms_norm`` / ``RMSNorm`` with
second-order gradients, ``layer_norm`` / ``LayerNorm``). Importing the package
loads nothing; the library is loaded on first use and a missing library is an
error.
"""
