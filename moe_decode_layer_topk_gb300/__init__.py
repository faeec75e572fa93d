"""GB300-native mixture-of-experts decode-layer forward (router, top-k routing,
FP4 experts, shared-expert blend) behind a C ABI (include/moe.h)."""
