"""GB300-native FLARE++ mixer forward.

``rank_latent_routing_gb300.flarepp`` binds the C-ABI library (CUDA kernels for
sm_103a); ``rank_latent_routing_gb300.workloads`` draws seeded synthetic inputs.
Importing the package loads neither.
"""
