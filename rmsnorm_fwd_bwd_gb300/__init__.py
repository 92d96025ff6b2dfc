"""RMSNorm forward/backward for one GB300 (sm_103a).

The compute path is the C-ABI library ``librmsnorm.so`` built from ``csrc/``;
``binding`` is its thin Python front end. Importing the package loads nothing;
the library is loaded on first use and a missing library is an error.
"""
