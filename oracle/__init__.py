"""fp64 CPU oracle of the Gated-DeltaNet mixer. Test infrastructure only: the
product path (the CUDA library and its binding) never imports this package."""
