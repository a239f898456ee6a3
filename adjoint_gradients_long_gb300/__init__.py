"""GB300-native adjoint-sharding gradient path for residual stacks of diagonal selective SSM layers.

The compute path lives in the CUDA library ``libadj.so`` (C ABI declared in
``include/adj.h``); ``adjoint_gradients_long_gb300.lib`` marshals arguments to it.
Importing this package loads nothing; the library is opened on first use.
"""
